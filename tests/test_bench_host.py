"""bench.py's host-side arithmetic and records (CPU only): algorithmic byte
counts against hand-counted values, and the traffic records' source hashes."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_prefill_bytes_by_hand():
    b = load_bench()
    # one token-head at d = 128: q, k, b, log_decay (4 x 128 x 2 B), v, w (2 x 128 x 2 B), fp32 o (128 x 4 B)
    assert b.prefill_bytes(1, 1, 1, 128, 128, s0=False, st=False) == 1024 + 512 + 512
    # the GDN-2 layer call: 262,144 token-heads plus S_T (64 heads x 64 KB)
    assert b.prefill_bytes(4, 4096, 16, 128, 128) == 262144 * 2048 + 64 * 65536
    assert b.prefill_bytes(4, 4096, 16, 128, 128) == 541065216


def test_backward_and_decode_bytes_by_hand():
    b = load_bench()
    # per token-head: six bf16 inputs (1536 B), fp32 do (512 B), six fp32 gradients (3072 B)
    assert b.backward_bytes(1, 1, 1, 128, 128) == 1536 + 512 + 3072 + 65536
    assert b.backward_bytes(4, 4096, 16, 128, 128) == 1346371584
    # per head-step: fp32 state read + written (2 x 64 KB), six bf16 inputs, fp32 o
    assert b.decode_bytes(1, 1, 128, 128) == 131072 + 1536 + 512


def test_traffic_records_name_existing_sources_and_captures():
    b = load_bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    assert {"prefill_gdn2_layer_T4096", "decode_B256_H16_d128", "prefill_long_T65536",
            "backward_gdn2_layer_T4096"} <= set(rec)
    for key, r in rec.items():
        assert b.kernel_source_hash(r["sources"]) is not None, key
        assert os.path.exists(os.path.join(ROOT, r["capture"])), key
        assert r["dram_bytes_per_launch"] > 0, key
        if "per_kernel" in r:
            assert sum(r["per_kernel"].values()) == r["dram_bytes_per_launch"], key


def test_packed_offsets_partition_the_rows():
    """The packed-sequence leg's offsets: seeded, n strictly increasing ranges that
    cover every row once, lengths not all multiples of the 64-token chunk."""
    b = load_bench()
    cu = b.packed_offsets(16384, 8)
    assert cu.dtype.is_floating_point is False and cu.numel() == 9
    assert int(cu[0]) == 0 and int(cu[-1]) == 16384
    lengths = (cu[1:] - cu[:-1]).tolist()
    assert all(L > 0 for L in lengths) and sum(lengths) == 16384
    assert any(L % 64 for L in lengths)
    assert b.packed_offsets(16384, 8).tolist() == cu.tolist()


def test_cpu_baseline_reports_one_thread_times():
    """The oracle baseline on a small synthetic problem (CPU only): its record
    carries the sampled rate and the one-thread times of one head and of the tiny
    fp32 workload."""
    import torch

    from gated_delta_rule_166_b300.inputs import make_prefill_inputs

    b = load_bench()
    x = make_prefill_inputs(1, 64, 2, 32, 32, dtype=torch.bfloat16, seed=3)
    rec = b.cpu_baseline(x, budget_s=0.01)
    assert rec["kind"] == "oracle" and rec["value"] > 0 and rec["cores"] >= 1
    assert set(rec["one_thread_s"]) == {"gdn2_layer_T4096_one_head", "tiny_f32"}
    assert all(v > 0 for v in rec["one_thread_s"].values())
