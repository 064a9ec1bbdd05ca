"""The benchmark's work model (the numerators of every rate and roofline fraction), on CPU.

Effective attention FLOP = 4 * head_dim * Hq * (query-key pairs the mask keeps); prep and decode
bytes are algorithmic (each input read once, each output written once). The pair count is
checked against a dense-mask brute force, and the full-size figures against the closed forms
for one 16384-token request: sum_p min(p + 1, 1024) = 1024 * 1025 / 2 + 15360 * 1024 pairs
under window_left 1023, and 16384 * 16385 / 2 pairs fully causal.
"""
import os
import sys

import numpy as np

import brute
from paged_sliding_window_qkv_gb300 import workloads as W

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_visible_pairs_match_a_dense_mask():
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(20):
        R = int(rng.integers(1, 4))
        lens = rng.integers(1, 30, R)
        starts = rng.integers(0, 40, R)
        b = W.make_batch(rng, lens, starts, 8)
        for window in (-1, 0, 3, 17):
            want = 0
            for r in range(R):
                pos = [int(starts[r]) + t for t in range(int(lens[r]))]
                m = brute.dense_mask(pos, int(starts[r] + lens[r]), window)
                want += sum(map(sum, m))
            assert bench.visible_pairs(b, window) == want


def test_full_size_figures_match_their_closed_forms():
    wl5 = W.make_workload(5)
    hd256, hd512 = wl5.families
    pairs256 = 1024 * 1025 // 2 + (16384 - 1024) * 1024
    pairs512 = 16384 * 16385 // 2
    assert bench.visible_pairs(hd256.batch, 1023) == pairs256 == 16_253_440
    assert bench.visible_pairs(hd512.batch, -1) == pairs512 == 134_225_920
    assert bench.attn_flops(hd256) == 4 * 256 * 16 * pairs256        # 2.663e11
    assert bench.attn_flops(hd512) == 4 * 512 * 16 * pairs512        # 4.398e12
    # prep: per token, hd256 moves 16 q + 8 k + 8 v rows in and 16 q + 8 k + 8 v rows out of
    # 512 B, a 1 KB rotary row and a 4 B request index; hd512 16 q + 1 k in, 16 q + 1 k + 1 v out
    # of 1 KB, a 2 KB rotary row and 4 B
    assert bench.prep_bytes(hd256) == 16384 * (64 * 512 + 1024 + 4) == 553_713_664
    assert bench.prep_bytes(hd512) == 16384 * (35 * 1024 + 2048 + 4) == 620_822_528


def test_decode_bytes_count_every_visible_row_once():
    wl4 = W.make_workload(4)
    for fi in wl4.families:
        f, b = fi.family, fi.batch
        rows = 0
        for r in range(b.num_req):
            p = int(b.start_pos[r])
            lo = max(0, p - f.window_left) if f.window_left >= 0 else 0
            rows += p + 1 - lo
        want = (rows * f.num_kv_heads * f.head_dim * 2 * 2          # K and V rows, bf16
                + b.num_req * f.num_qo_heads * f.head_dim * 2 * 2    # q in, out written
                + (rows // b.page_size + b.num_req) * 4)             # page ids of the visible keys
        assert bench.decode_bytes(fi) == want


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    # a call's DRAM bytes come from the committed capture only while its kernel source hashes
    # as recorded; any edit of the source (or a missing entry or file) gives None
    import hashlib
    import json
    csrc = tmp_path / "paged_sliding_window_qkv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_bytes(b"kernel v1\n")
    entry = {"case": "c", "source": "k.cu", "sha256": hashlib.sha256(b"kernel v1\n").hexdigest(),
             "dram_bytes_per_launch": 12345, "scaled": 1}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"calls": {"call": entry}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("call") == 12345
    assert bench.kernel_traffic("other call") is None
    src.write_bytes(b"kernel v2\n")
    assert bench.kernel_traffic("call") is None
    src.unlink()
    assert bench.kernel_traffic("call") is None

