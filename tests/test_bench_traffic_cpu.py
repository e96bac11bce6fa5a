"""bench.py reports the committed ncu DRAM traffic of a family only for the
workload it was taken on: the current kernel sources (source hash) and the
same algorithmic bytes per step (a run restricted by --only has fewer)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _recorded(family):
    vals = {}
    for line in open(os.path.join(ROOT, "profiles", f"{family}_traffic.txt")):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    return vals


def test_traffic_only_for_the_recorded_workload():
    b = _bench()
    for fam in ("qmv", "qmm_t", "q8_0", "q4_k"):
        vals = _recorded(fam)
        alg = int(vals["algorithmic_bytes_per_step"])
        current = vals["source_sha256_16"] == b.source_hash(b.KERNEL_SOURCES[fam])
        got = b.recorded_traffic(fam, alg)
        assert got == (float(vals["dram_bytes_per_step"]) if current else None), fam
        assert b.recorded_traffic(fam, alg // 8) is None, fam   # a restricted run


def test_step_bytes_match_the_recorded_families():
    """The families' algorithmic bytes per step, as bench.py counts them,
    are the ones the traffic summaries were recorded for."""
    b = _bench()
    per_family = {
        "qmv": sum(b.affine_bytes(1, N, K) for (N, K) in b.QMV_SHAPES),
        "qmm_t": sum(b.affine_bytes(M, N, K) for (K, N, M) in b.QMM_SHAPES),
        "q8_0": sum(b.q8_bytes(N, K) for (N, K) in b.BLOCKQ_SHAPES),
        "q4_k": sum(b.q4k_bytes(N, K) for (N, K) in b.BLOCKQ_SHAPES),
    }
    for fam, alg in per_family.items():
        assert int(_recorded(fam)["algorithmic_bytes_per_step"]) == alg, fam
    assert per_family == b.step_bytes()
    assert sum(per_family.values()) == 514569216   # the step's bytes as the bench line reports them
