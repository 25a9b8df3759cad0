"""Host-side logic of bench.py (no GPU): the algorithmic work behind the
roofline and the TFLOP/s metric, the oracle sample's flop count, the clock
record parser and the ncu traffic table lookup.

The flop totals are checked against the closed form of one layer written out
here: Q/K/V, output, gate/up and down projections 2*T*(h*(h + 2hk) + h*h +
3*h*F) (with hk = h: T*(8h^2 + 6hF)) plus causal attention 4*B*H*dh*S(S+1)/2,
the triangle only.  The backward's model flops are twice the forward's.
"""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from folded_tensor_sequence_gb300.configs import BY_NAME  # noqa: E402


def closed_form_fwd(B, S, h, H, dh, F, hk):
    T = B * S
    linear = 2 * T * h * (h + 2 * hk) + 2 * T * h * h + 2 * T * h * 2 * F + 2 * T * F * h
    attention = 4 * B * H * dh * S * (S + 1) // 2
    return linear + attention


FWD_STEPS = ("QKV projection", "attention", "output projection", "gate/up projection", "down projection")
BWD_STEPS_FUSED = ("dM = dY Wd^T", "dW_down", "dH", "dW_gate_up", "dO", "dW_O", "attention bwd fused", "dx",
                   "dW_QKV")
BWD_STEPS_SPLIT = ("dM = dY Wd^T", "dW_down", "dH", "dW_gate_up", "dO", "dW_O", "attention bwd dK/dV",
                   "attention bwd dQ", "dx", "dW_QKV")


def fwd_cfgs():
    return [c for c in BY_NAME.values() if not c.decode]


@pytest.mark.parametrize("cfg", fwd_cfgs(), ids=lambda c: c.name)
def test_forward_work_sums_to_the_closed_form(cfg):
    w = bench.step_work(cfg)
    total = sum(w[k][0] for k in FWD_STEPS)
    assert total == closed_form_fwd(cfg.batch, cfg.seq, cfg.hidden, cfg.heads, cfg.head_dim, cfg.ffn,
                                     cfg.kv_hidden)
    assert total == cfg.fwd_flops()
    # permutes move bytes, no flops
    assert w["zigzag permute"][0] == 0 and w["zigzag permute"][1] == 2 * cfg.batch * cfg.seq * cfg.hidden * (
        2 if cfg.dtype == "bf16" else 4)


@pytest.mark.parametrize("det", [False, True], ids=["fused", "split"])
@pytest.mark.parametrize("cfg", [c for c in fwd_cfgs() if c.backward], ids=lambda c: c.name)
def test_training_work_is_three_forwards(cfg, det):
    w = bench.step_work(cfg, det)
    fwd = sum(w[k][0] for k in FWD_STEPS)
    bwd = sum(w[k][0] for k in (BWD_STEPS_SPLIT if det else BWD_STEPS_FUSED))
    assert bwd == 2 * fwd
    assert fwd + bwd == 3 * cfg.fwd_flops()


def test_headline_flops_match_the_table():
    # D=8, B=2, S=16384, h=4096, F=14336: linear 15.94 TFLOP + attention 4.40 TFLOP
    c = BY_NAME["bf16_D8_b2_s16384_h4096"]
    w = bench.step_work(c)
    linear = sum(w[k][0] for k in FWD_STEPS if k != "attention")
    assert abs(linear - 15.94e12) / 15.94e12 < 1e-3
    assert abs(w["attention"][0] - 4.40e12) / 4.40e12 < 1e-3
    assert abs(c.fwd_flops() - 20.34e12) / 20.34e12 < 1e-3


def test_oracle_sample_of_the_whole_sequence_is_one_sequence_forward():
    for cfg in fwd_cfgs():
        assert bench.sample_flops(cfg, cfg.seq) == cfg.with_(batch=1).fwd_flops()
    # a prefix: projections scale with the tokens, attention with the causal triangle
    c = BY_NAME["bf16_D8_b2_s16384_h4096"]
    p = 512
    assert bench.sample_flops(c, p) == closed_form_fwd(1, p, c.hidden, c.heads, c.head_dim, c.ffn, c.kv_hidden)


def test_decode_work_streams_every_weight_once():
    for cfg in (c for c in BY_NAME.values() if c.decode):
        w = bench.step_work(cfg)
        h, F, hk, B = cfg.hidden, cfg.ffn, cfg.kv_hidden, cfg.batch
        W3 = h + 2 * hk
        cache = 2 * B * cfg.seq * hk * 2                    # K and V rows of every cached position
        tokens = B * (h + W3 + 2 * h + 3 * h + h + F + F + 2 * h) * 2  # each step's token vectors in and out
        weights = sum(w[k][1] for k in w) - cache - tokens
        assert weights == (h * W3 + h * h + 2 * F * h + h * F) * 2  # every packed weight once
        assert weights > 0.99 * (sum(w[k][1] for k in w) - cache)  # the tokens are a rounding error


class _Done:
    def terminate(self):
        pass

    def wait(self):
        pass


def test_clock_parser_reads_median_and_reasons(tmp_path):
    lines = [
        "0, 1800, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1900, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2070, 990.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = bench.ClockSampler("0")
    s.proc = _Done()
    s.out = open(tmp_path / "clk.csv", "w+")
    s.out.write("\n".join(lines) + "\n")
    got = s.summary()
    assert got["sm_mhz"] == 1900.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] == 3
    s.out.close()
    none = bench.ClockSampler("0").summary()
    assert none["sm_mhz"] is None and none["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_lookup_needs_the_same_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {("step", "wl"): (123.0, str(src), sha)})
    assert bench.ncu_traffic("step", "wl") == 123.0
    assert bench.ncu_traffic("step", "other") is None
    src.write_text("// kernel v2\n")
    assert bench.ncu_traffic("step", "wl") is None


def test_traffic_table_names_existing_sources_and_steps():
    for (step, workload), (value, path, sha) in bench.NCU_TRAFFIC.items():
        assert workload in BY_NAME and value > 0 and len(sha) == 16
        assert os.path.exists(os.path.join(ROOT, path))
        assert (step in bench.step_work(BY_NAME[workload])
                or step.removesuffix(" (standalone)") in bench.LAYOUT_STEPS), step


def test_nominal_peak_is_the_clock_derived_tensor_rate():
    # 8192 flops per SM cycle (one 128 x 256 x 16 bf16 MMA every 128 cycles) x 152 SMs x clock
    assert bench.nominal_bf16_tflops(152, 2070.0) == pytest.approx(8192 * 152 * 2.07e9 / 1e12)
    assert bench.nominal_bf16_tflops(152, 2070.0) == pytest.approx(2577.5, abs=0.1)
    # at about 1.8 GHz it is the 2.25 PFLOP/s nominal figure
    assert bench.nominal_bf16_tflops(152, 1807.0) == pytest.approx(2250.0, rel=1e-3)
    assert bench.nominal_bf16_tflops(152, None) is None


def test_host_description_names_cpus_and_model():
    h = bench.host_cpu()
    assert h["nproc"] == os.cpu_count() and h["nproc"] >= 1
    assert isinstance(h["cpu_model"], str) and h["cpu_model"]
    assert h["machine"]
