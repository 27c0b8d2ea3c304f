"""Failure detection on the GPU without a fault: the bounded mbarrier wait that every fused
kernel uses gives up after its limit and reports GDN_DEV_TIMEOUT in the status word instead of
hanging (gdn_selftest_wait_timeout runs it in a one-thread kernel with no copy or MMA in
flight, on an mbarrier that nobody arrives on), and the context stays usable afterwards."""
import pytest
import torch

from chunked_gated_delta_gdn_gb300 import _lib, gated_delta_decode, synthetic

pytestmark = pytest.mark.gpu


def selftest(limit_ns, arrive_first):
    lib = _lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.gdn_selftest_wait_timeout(st.data_ptr(), limit_ns, arrive_first, waited.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.GDN_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    return int(st.item()), int(waited.item())


def test_wait_on_an_mbarrier_nobody_arrives_on_times_out_and_reports():
    bits, waited = selftest(10_000, arrive_first=0)          # 10 us limit
    print("timed-out wait returned after %d ns, status 0x%x" % (waited, bits))
    assert bits & _lib.GDN_DEV_TIMEOUT
    assert 10_000 <= waited < 10_000_000                      # gave up, and soon after its limit


def test_wait_on_a_completed_phase_succeeds_without_a_report():
    bits, waited = selftest(10_000_000, arrive_first=1)
    assert bits == 0
    assert waited < 1_000_000


def test_context_usable_after_a_timeout():
    selftest(10_000, arrive_first=0)
    d = synthetic.decode_inputs(n=4, Hqk=1, Hv=2, K=128, V=128, dtype=torch.bfloat16,
                                num_slots=6, pad_frac=0.0, seed=5)
    o = gated_delta_decode(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.g.cuda(), d.beta.cuda(),
                           d.ssm_state.cuda(), d.batch_indices.cuda(), check=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()


def test_limits_are_validated_on_the_host():
    lib = _lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.gdn_selftest_wait_timeout(None, 1000, 0, None, None) == _lib.GDN_ERR_NULL
    assert lib.gdn_selftest_wait_timeout(st.data_ptr(), 0, 0, None, None) == _lib.GDN_ERR_SHAPE
    assert lib.gdn_selftest_wait_timeout(st.data_ptr(), 10**9, 0, None, None) == _lib.GDN_ERR_SHAPE
