"""bench.py's roofline arithmetic on the host (no GPU): the minimal-traffic byte counts, the
choice of the bound, the fractions, and the traffic figure's tie to the kernel sources."""
import pytest

import bench
import synth

# Minimal traffic (each input read once, each output written once, fp32) of the workloads:
# 4*(4*BTD + 2*BTN + Di*N + Di) for the forward, 4*(7*BTD + 4*BTN + 2*Di*N + 2*Di) for the
# backward, worked out by hand from the shapes.
MINIMAL = {
    "mamba130m": (202_479_616, 354_627_584, 557_107_200),
    "mamba370m": (539_107_328, 943_996_928, 1_483_104_256),
    "mamba1p4b": (538_198_016, 942_178_304, 1_480_376_320),
    "longseq": (2_718_574_592, 4_766_060_544, 7_484_635_136),
}


@pytest.mark.parametrize("name", sorted(MINIMAL))
def test_minimal_bytes(name):
    mb = bench.minimal_bytes(synth.BY_NAME[name])
    assert (mb["fwd"], mb["bwd"], mb["total"]) == MINIMAL[name]


def test_roofline_bound_and_fractions():
    w = synth.BY_NAME["longseq"]
    r = bench.roofline_of(w, fwd_s=3.66e-3, bwd_s=8.70e-3, step_s=12.33e-3, sm_mhz=2070.0,
                          hbm_gbs=6783.1, hbm_source="measured")
    # d_state 64: the fp32 floor of the backward call is far above its HBM floor
    assert r["bound"] == "alu"
    ns = w.btd * w.d_state
    alu = bench.BWD_FP32_OPS_PER_ELEMENT_STATE * ns / 8.70e-3 / 1e9
    assert r["achieved"] == pytest.approx(alu)
    assert r["peak"] == pytest.approx(152 * 128 * 2.070)
    assert r["frac"] == pytest.approx(alu / (152 * 128 * 2.070))
    assert r["hbm"]["frac"] == pytest.approx(4_766_060_544 / 8.70e-3 / 1e9 / 6783.1)
    assert r["hbm_frac_step"] == pytest.approx(7_484_635_136 / 12.33e-3 / 1e9 / 6783.1)
    assert r["algorithmic_bytes_per_launch"] == 4_766_060_544


def test_traffic_only_while_the_sources_match(monkeypatch):
    w = synth.BY_NAME["mamba370m"]
    args = dict(fwd_s=2.4e-4, bwd_s=5.2e-4, step_s=7.4e-4, sm_mhz=2070.0, hbm_gbs=6783.1,
                hbm_source="measured")
    cap = bench.BWD_TRAFFIC_CAPTURES["mamba370m"]
    monkeypatch.setattr(bench, "kernel_digest", lambda: cap[1])
    assert bench.roofline_of(w, **args)["traffic"] == cap[0]
    monkeypatch.setattr(bench, "kernel_digest", lambda: "0" * 16)
    r = bench.roofline_of(w, **args)
    assert r["traffic"] is None and r["traffic_capture"] is None
