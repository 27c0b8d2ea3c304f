"""Host-side pieces of bench.py (CPU only): the code hash that keys the committed DRAM-traffic
record (the kernel source and the local headers it includes), and the record lookup itself."""
import json
import os

import bench

KERNEL = """// a kernel
__global__ void k(float* x) {   /* body */
  x[threadIdx.x] = 1.f;  // one store
}
"""


def write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return str(p)


def test_comment_and_whitespace_edits_keep_the_code_hash(tmp_path):
    a = bench.kernel_code_hash(write(tmp_path, "a.cu", KERNEL))
    edited = KERNEL.replace("// one store", "// the only store").replace("/* body */", "/*\n multi\n line */")
    b = bench.kernel_code_hash(write(tmp_path, "b.cu", edited.replace("  x[", "    x[")))
    assert a == b


def test_code_edits_change_the_code_hash(tmp_path):
    a = bench.kernel_code_hash(write(tmp_path, "a.cu", KERNEL))
    b = bench.kernel_code_hash(write(tmp_path, "b.cu", KERNEL.replace("1.f", "2.f")))
    c = bench.kernel_code_hash(write(tmp_path, "c.cu", KERNEL.replace("x[threadIdx.x]", "x[threadIdx.y]")))
    assert len({a, b, c}) == 3


def test_traffic_record_is_null_unless_the_code_matches(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    src = tmp_path / "chunked_gated_delta_gdn_gb300" / "csrc"
    prof.mkdir()
    src.mkdir(parents=True)
    (src / "gdn_chunk_tc.cu").write_text(KERNEL)
    rec = {"kernel_code_sha256_16": bench.kernel_code_hash(str(src / "gdn_chunk_tc.cu")),
           "dram_bytes_per_full_launch": 1234}
    (prof / "chunk_tc_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record() == 1234
    (src / "gdn_chunk_tc.cu").write_text(KERNEL + "// a comment\n")
    assert bench.traffic_record() == 1234
    (src / "gdn_chunk_tc.cu").write_text(KERNEL.replace("1.f", "3.f"))
    assert bench.traffic_record() is None
    os.remove(prof / "chunk_tc_traffic.json")
    assert bench.traffic_record() is None


def test_header_edits_change_the_code_hash_and_void_the_record(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    src = tmp_path / "chunked_gated_delta_gdn_gb300" / "csrc"
    prof.mkdir()
    src.mkdir(parents=True)
    header = "// tile sizes\nconstexpr int kBox = 64;\n"
    (src / "tiles.cuh").write_text(header)
    (src / "gdn_chunk_tc.cu").write_text('#include "tiles.cuh"\n#include <cuda.h>\n' + KERNEL)
    rec = {"kernel_code_sha256_16": bench.kernel_code_hash(str(src / "gdn_chunk_tc.cu")),
           "dram_bytes_per_full_launch": 99}
    (prof / "chunk_tc_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record() == 99
    (src / "tiles.cuh").write_text(header.replace("// tile sizes", "// box edge"))
    assert bench.traffic_record() == 99            # comment edit in the header: still current
    (src / "tiles.cuh").write_text(header.replace("64", "128"))
    assert bench.traffic_record() is None          # code edit in the header: stale
