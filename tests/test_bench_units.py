"""The benchmark's units of work: algorithmic bytes and flops per launch, as
defined for the hot path's measurement, checked against the figures worked
out by hand for each workload (N*K/2 packed weight bytes, N*K/16 scale
bytes, activation and output bytes, bias, the 4-byte global scale)."""

import bench


def test_gemv_bytes():
    # M = 4, N = K = 5120: 13,107,200 + 1,638,400 + 40,960 + 40,960 + 4
    assert bench.gemv_bytes(4, 5120, 5120) == 14_827_524
    assert bench.gemv_bytes(1, 5120, 5120) == 14_766_084
    assert bench.gemv_bytes(8, 5120, 5120) == 14_909_444
    # lm_head: 389,283,840 + 48,660,480 + 40,960 + 1,216,512 + 304,128 (bias) + 4
    assert bench.gemv_bytes(4, 152064, 5120, bias=True) == 439_505_924


def test_fp8_gemv_bytes():
    # N = K = 5120, bs = 128: 26,214,400 + 4 * 5120 * 40 + 2 * 4 * 5120 * 2
    assert bench.gemv_bytes(4, 5120, 5120, 128, kind="fp8") == 26_214_400 + 819_200 + 81_920


def test_dequant_and_actq_bytes():
    # N = 17408, K = 5120: 44,564,480 + 5,570,560 + 178,257,920 + 4
    assert bench.dequant_bytes(17408, 5120) == 228_392_964
    # M = 8192, K = 5120: 83,886,080 read + 20,971,520 codes + 2,621,440 scales
    assert bench.actq_bytes(8192, 5120) == 107_479_040


def test_prefill_flops():
    assert 2 * 8192 * 17408 * 5120 == 1_460_288_880_640


def test_recorded_traffic_matches_current_sources():
    """The DRAM bytes the bench line reports for the headline kernel come from
    a committed ncu record keyed by a hash of that kernel's sources; the
    record must have been taken on the sources as they stand (a kernel change
    needs a new capture), and it must equal the algorithmic bytes within 1 %
    (no re-reads) for the figure to mean what the line says."""
    t = bench.recorded_traffic("gemv_decode_M4_N5120_K5120")
    assert t is not None, "profiles/ncu_traffic.json predates the current GEMV sources"
    alg = bench.gemv_bytes(4, 5120, 5120)
    assert abs(t - alg) / alg < 0.01
