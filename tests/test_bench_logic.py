"""Host logic of bench.py that turns a run into the roofline fields: the
algorithmic bytes of a step, which kernel's ncu summary its traffic comes
from, how many kernels a step launches, and when a committed summary is
trusted.  No GPU is needed."""

import bench


def test_headline_step_bytes():
    """B = 1, H = 64, per-tensor FP8 cache, worked out from the shapes: W_QB
    64*192*1536*2 = 37,748,736; W_UK 64*128*512*2 = 8,388,608; gammas
    (1536+512)*2 = 4,096; q_a, kv_c, k_pe and the slot 4,232; q_latent and
    q_pe 64*576*2 = 73,728; q_c 3,072; one 576-byte cache row."""
    want = 37_748_736 + 8_388_608 + 4_096 + 4_232 + 73_728 + 3_072 + 576
    assert want == 46_223_048
    assert bench.algorithmic_bytes(1, 64, 0) == want


def test_step_bytes_grow_by_layout_and_hidden_row():
    base = bench.algorithmic_bytes(8, 128, 0)
    # the cache rows differ by layout only: 576, 656, 352 bytes per token
    assert bench.algorithmic_bytes(8, 128, 1) - base == 8 * (656 - 576)
    assert bench.algorithmic_bytes(8, 128, 2) - base == 8 * (352 - 576)
    # from the hidden row: W_QKV_A 2112*7168*2, the hidden rows, the fused row
    assert (bench.algorithmic_bytes(8, 128, 0, hidden=True) - base ==
            2112 * 7168 * 2 + 8 * 7168 * 2 + 8 * 2112 * 2)


def test_dominant_kernel():
    assert bench.dominant_kernel("mla_absorb_pair_kernel<8>") == "mla_absorb_pair_kernel<8>"
    assert bench.dominant_kernel("mla_wide_norm_kernel+mla_wide_kernel") == "mla_wide_kernel"
    assert bench.dominant_kernel("mla_absorb_kernel<1>+mla_close_kernel<1>") == "mla_absorb_kernel<1>"


def test_launches_per_step():
    # wide: both kernels once per 64 tokens
    assert bench.launches_per_step("mla_wide_norm_kernel+mla_wide_kernel", 64) == 2
    assert bench.launches_per_step("mla_wide_norm_kernel+mla_wide_kernel", 65) == 4
    # the 16-token paired kernel once per 16 tokens above 16
    assert bench.launches_per_step("mla_absorb_pair_kernel<16>", 16) == 1
    assert bench.launches_per_step("mla_absorb_pair_kernel<16>", 40) == 3
    # from the hidden row: the qkv_a projection once per 8 tokens first
    assert bench.launches_per_step("mla_absorb_pair_kernel<8>", 1, hidden=True) == 2
    assert bench.launches_per_step("mla_absorb_pair_kernel<16>", 9, hidden=True) == 3


def test_traffic_only_from_a_summary_of_the_current_sources(monkeypatch):
    name = bench.profile_name("mla_absorb_pair_kernel<8>", "latency_b1_h64_e4m3")
    assert name.endswith("profiles/mla_absorb_pair_kernel_latency_b1_h64_e4m3.txt")
    # a summary taken on other sources (another hash) gives no traffic
    monkeypatch.setattr(bench, "kernel_hash", lambda kernel: "0" * 16)
    assert bench.read_traffic("mla_absorb_pair_kernel<8>", "latency_b1_h64_e4m3") is None
    # nor does a workload without a summary
    assert bench.read_traffic("mla_absorb_pair_kernel<8>", "no_such_workload") is None
