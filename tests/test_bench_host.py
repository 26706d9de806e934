"""Host-side logic of the benchmark, on the CPU: the algorithmic work that the
roofline fractions divide by, the fraction arithmetic, the per-kernel spans
taken from kernel-boundary events, and the rule that a DRAM-traffic figure is
reported only for the kernel source it was measured on."""

import pytest

import bench
import synth


TRAIN = synth.Shape(T=49152, D=768, H=6, d_qk=96, d_v=128, seq_len=8192)


def test_algorithmic_work_at_the_training_shape():
    w = bench.algorithmic_work(TRAIN)
    T, D, H, N = 49152, 768, 6, 1920
    # the packed output width: H heads of 96 + 96 + 128 columns
    assert TRAIN.N == N
    assert w["bank_refresh"] == ("hbm", N * D * 2 + 2 * N * D)         # one bf16 read, both code layouts
    assert w["x_quant"] == ("hbm", 2 * T * D * 2 + T * D)              # x twice, x8 once
    for g in ("fwd_gemm", "dx_gemm", "dw_gemm"):
        assert w[g] == ("tensor", 2.0 * T * D * N)                     # 144.96 GFLOP each
    q = H * T * 96 * 2                                                 # one of q, k, dq, dk (bf16)
    v = H * T * 128 * 2                                                # one of v, dv
    bwd_in = 4 * q + v + 2 * H * T * 4 + T * 4                         # + rstd, pos
    assert w["dy_amax"] == ("hbm", bwd_in)
    assert w["dy_quant"] == ("hbm", bwd_in + T * N)                    # + dY8 codes
    assert abs(w["fwd_gemm"][1] - 144.96e9) < 0.01e9
    assert abs(w["dy_amax"][1] - 304.6e6) < 0.1e6
    assert abs(w["dy_quant"][1] - 398.9e6) < 0.1e6
    assert set(w) == set(bench.KERNELS)


def test_kernel_table_fractions():
    peaks = dict(hbm=6000.0, bf16=1500.0, bf16_sus=1200.0)
    work = {"a": ("hbm", 6.0e9), "b": ("tensor", 3.0e12)}
    # 1 ms for 6 GB = 6000 GB/s (the whole HBM peak); 3 TFLOP in 1 ms = 3000
    # TFLOP/s against the E4M3 peak of 2 x 1500 (the burst bf16 figure: the
    # timed regions last milliseconds)
    kt = bench.kernel_table({"a": 1.0, "b": 1.0}, work, peaks)
    assert kt["a"]["unit"] == "GB/s" and kt["a"]["achieved"] == pytest.approx(6000.0)
    assert kt["a"]["frac"] == pytest.approx(1.0)
    assert kt["b"]["unit"] == "TFLOP/s" and kt["b"]["achieved"] == pytest.approx(3000.0)
    assert kt["b"]["frac"] == pytest.approx(1.0)
    kt = bench.kernel_table({"a": 2.0, "b": 4.0}, work, peaks)
    assert kt["a"]["frac"] == pytest.approx(0.5) and kt["b"]["frac"] == pytest.approx(0.25)


class _Ev:
    """Stand-in for a recorded CUDA event: a time stamp in ms."""

    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_span_means_from_boundary_events():
    assert len(bench.SPANS) == len(bench.KERNELS)
    assert all(0 <= a < b < bench.EVENTS_PER_STEP for a, b in bench.SPANS)
    # two steps; event i at time i * (step + 1) ms, so every span of step s
    # lasts (b - a) * (s + 1) ms and the mean over both is 1.5 * (b - a)
    steps = [[_Ev(i * (s + 1.0)) for i in range(bench.EVENTS_PER_STEP)] for s in range(2)]
    per = bench.span_means(steps, bench.KERNELS, bench.SPANS)
    for name, (a, b) in zip(bench.KERNELS, bench.SPANS):
        assert per[name] == pytest.approx(1.5 * (b - a))


def test_traffic_only_for_the_measured_source(monkeypatch):
    T0 = bench.TRAFFIC["T"]
    fake = {"T": T0, "sources_sha256": {"bwd": bench.sources_sha256("bwd"), "gemm": "0" * 64},
            "bytes": {"dy_amax": ("bwd", 100.0e6), "fwd_gemm": ("gemm", 50.0e6)}}
    monkeypatch.setattr(bench, "TRAFFIC", fake)
    # scaled by the tokens when the source matches the capture
    assert bench.traffic_for("dy_amax", 2 * T0) == round(200.0e6)
    # a kernel whose source changed since the capture, or one never captured
    assert bench.traffic_for("fwd_gemm", T0) is None
    assert bench.traffic_for("x_quant", T0) is None


def test_job_throughput_and_slowest_rank():
    # one process: the job's time is this rank's
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    # every rank's tokens over the slowest rank's time
    assert bench.job_tokens_per_s(49152, 4, 0.5) == pytest.approx(4 * 49152 / 0.5e-3)
