"""The measurement arithmetic of bench.py, on CPU: algorithmic work per
launch, the roofline object built from a profile, the traffic table lookup
and the dominant-kernel choice.  No GPU and no timing involved."""
import pytest

import bench
from dictionary_sparse_kv_gb300 import synthetic as S

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def test_kernel_work_per_launch():
    w = S.WORKLOADS["decode_3b"]                 # 56 dictionaries, N=4096, d=128, n=256, s=8
    V = w.V
    nv = w.G * V
    bound, work, unit = bench.kernel_work(w, "screen", V)
    assert (bound, unit) == ("hbm", "GB/s")
    assert work == 56 * 4096 * 128 * 2 + nv * 128 * 2        # dictionaries once + inputs
    bound, work, unit = bench.kernel_work(w, "greedy", V)
    assert (bound, unit) == ("hbm", "GB/s")
    # pool ids, scores, G_jj; 7 Gram rows at the 256 pool ids; x and 8 rows; codes
    assert work == (256 * 12 + 7 * 256 * 4 + 9 * 128 * 2 + 8 * 8 + 4) * nv
    bound, work, unit = bench.kernel_work(w, "greedy", V, coder="pl")
    assert (bound, unit) == ("hbm", "GB/s")
    assert work == (9 * 128 * 2 + 8.0 * 8 + 4.0) * nv        # s rows + x in, codes out
    _, topn_gm, _ = bench.kernel_work(w, "topn", V)
    _, topn_pl, _ = bench.kernel_work(w, "topn", V, coder="pl")
    assert topn_gm - topn_pl == pytest.approx(8.0 * (256 - 8) * nv)   # the pool is s ids and scores for PL
    with pytest.raises(KeyError):
        bench.kernel_work(w, "nothing", V)


def test_roofline_from_profiles():
    w = S.WORKLOADS["decode_3b"]
    # (launches, total ms) per kernel class: the greedy dominates
    prof = {"screen": (10, 0.31), "topn": (20, 0.31), "greedy": (10, 2.27), "adapt": (10, 0.08)}
    timed = {"greedy": (20, 4.54)}
    roof, shares = bench.roofline(w, prof, timed, w.V, PEAKS, "measured", 152, 2070.0)
    assert roof["kernel"] == "greedy" and roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    byts = (256 * 12 + 7 * 256 * 4 + 9 * 128 * 2 + 8 * 8 + 4) * w.G * w.V
    assert roof["launch_ms"] == pytest.approx(0.227)
    assert roof["achieved"] == pytest.approx(byts / 0.227e-3 / 1e9, rel=1e-3)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 6800.0, abs=1e-4)     # rounded to 4 places
    assert sum(v["share"] for v in shares.values()) == pytest.approx(1.0, abs=1e-3)
    assert shares["greedy"]["launches"] == 10
    # without a timed figure for the dominant kernel the profile's own is used
    roof2, _ = bench.roofline(w, prof, {}, w.V, PEAKS, "measured", 152, 2070.0)
    assert roof2["launch_ms"] == pytest.approx(0.227)
    # the PL coder's fit is HBM-bound work
    roof3, _ = bench.roofline(w, {"greedy": (10, 0.24)}, {}, w.V, PEAKS, "measured", 152, 2070.0, coder="pl")
    assert roof3["bound"] == "hbm" and roof3["source"] == "k_pl.cu"


def test_dominant_kernel_and_traffic_lookup():
    assert bench.dominant_kernel({}) is None
    assert bench.dominant_kernel({"a": (1, 0.5), "b": (3, 0.7)}) == "b"
    w = S.WORKLOADS["decode_3b"]
    t = bench.traffic_for("greedy", w)
    # the committed table matches the committed greedy source, or the lookup
    # says it does not know (never a stale number)
    assert t is None or t > 56 * 4096 * 128 * 2 * 0.5
    from dataclasses import replace
    assert bench.traffic_for("greedy", replace(w, name="no_such_workload")) is None


def test_workload_config_names_the_coder():
    w = S.WORKLOADS["decode_3b"]
    c = bench.workload_config(w, w.G * w.V)
    assert c["vectors_per_step"] == 7168 and "decode_3b" in c["workload"] and "greedy" in c["coder"]
    assert "PL" in bench.workload_config(w, 1, "pl")["coder"]
    assert bench.job_throughput(1, 20, 7168, 6.0) == pytest.approx(20 * 7168 / 0.006)


def test_step_roofline_bytes():
    """decode_3b: 56 MiB of dictionaries, 1.75 MiB of inputs, 84 B of codes
    per vector and 0.9 MiB of usage counts per step: about 8.6 KB per vector,
    the figure the scope table quotes."""
    w = S.WORKLOADS["decode_3b"]
    r = bench.step_roofline(w, 7168, 0.300, PEAKS)
    algo = 56 * 4096 * 128 * 2 + 7168 * 128 * 2 + 7168 * (8 * 8 + 12) + 56 * 4096 * 4
    assert r["algorithmic_bytes"] == algo
    assert 8500 < r["bytes_per_vector"] < 8800
    assert r["frac"] == pytest.approx(algo / 0.3e-3 / 1e9 / 6800.0, abs=1e-4)


def test_screening_fractions():
    """Two launches per step of 2 x 65 536 vectors (the 16K prefill): HBM
    bytes = each launch's dictionaries + every input once; flops = 2 N d
    per vector."""
    w = S.WORKLOADS["prefill_3b_16k"]
    prof = {"screen": (8, 2.0)}                  # 4 steps, 2 launches each, 0.25 ms per launch
    r = bench.screening_fractions(w, prof, 4, PEAKS)
    flops = 2.0 * 4096 * 128 * 4 * 2 * 131072
    assert r["tensor"]["achieved_tflops"] == pytest.approx(flops / 2e-3 / 1e12, rel=1e-3)
    assert r["tensor"]["frac"] == pytest.approx(flops / 2e-3 / 1e12 / 1900.0, abs=1e-4)
    byts = 8 * 2 * 4096 * 128 * 2 + 4 * 2 * 131072 * 128 * 2
    assert r["hbm"]["achieved_gbs"] == pytest.approx(byts / 2e-3 / 1e9, rel=1e-3)
    assert bench.screening_fractions(w, {}, 4, PEAKS) is None


def test_traffic_from_ncu_csv(tmp_path):
    """Bytes per launch of one kernel from ncu's --csv rows (one row per
    launch and metric, units as ncu prints them)."""
    name = "void fadkv::(anonymous namespace)::greedy_gram_kernel<128, 1, 8, 8, true>(fadkv::Shape, fadkv::GramGreedyArgs)"
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
            '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')
    rows = [("0", name, "dram__bytes_read.sum", "Mbyte", "300.50"),
            ("0", name, "dram__bytes_write.sum", "Kbyte", "400"),
            ("1", "select_kernel", "dram__bytes_read.sum", "Mbyte", "29.4"),
            ("2", name, "dram__bytes_read.sum", "Gbyte", "0.3"),
            ("2", name, "dram__bytes_write.sum", "byte", "1,000")]
    lines = ["==PROF== Connected", head] + [
        f'"{i}","1","python","h","{k}","1","7","(128, 1, 1)","(1792, 1, 1)","0","10.3","m","{m}","{u}","{v}"'
        for i, k, m, u, v in rows]
    p = tmp_path / "t.csv"
    p.write_text("\n".join(lines) + "\n")
    byts, n = bench.traffic_from_ncu_csv(str(p), "greedy_gram_kernel")
    assert n == 2 and byts == pytest.approx(((300.5e6 + 400e3) + (0.3e9 + 1000)) / 2)
    with pytest.raises(ValueError):
        bench.traffic_from_ncu_csv(str(p), "no_such_kernel")
