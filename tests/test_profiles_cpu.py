"""The committed Nsight Compute summaries that bench.py reports from: present, parseable, and
consistent with the algorithmic bytes of the kernel they describe."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_tests", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_headline_algorithmic_bytes():
    """16 layers of H_kv=8, D=64, N=8192 mlx4g32 records (K and V), an S_suf=16 fp16 suffix,
    fp32 Q and O (+ one fp32 LSE per q head), H_q=32."""
    layers, H_q, H_kv, N, D, S = 16, 32, 8, 8192, 64, 16
    kv_dim = H_kv * D
    rec = kv_dim // 2 + (kv_dim // 32) * 2 * 2          # 4-bit codes + fp16 scale and bias per 32
    assert rec == 320
    per_layer = 2 * N * rec + 2 * H_kv * S * D * 2 + H_q * D * 4 + H_q * D * 4 + H_q * 4
    assert _bench().ALG_BYTES_STEP == layers * per_layer == 84_674_560


def test_headline_traffic_within_five_percent_of_algorithmic():
    b = _bench()
    t = b.traffic_from_profiles("decode_mlx4g32_gqa")
    assert t is not None, "the headline decode profile has no traffic_bytes_per_launch line"
    assert 1.0 <= t / b.ALG_BYTES_STEP <= 1.05, f"traffic {t:.0f} B vs algorithmic {b.ALG_BYTES_STEP} B"


def test_every_summary_names_its_command():
    names = sorted(f for f in os.listdir(PROFILES) if f.endswith((".txt", ".md")))
    assert names
    for f in names:
        text = open(os.path.join(PROFILES, f)).read()
        assert "ncu " in text and "--clock-control none" in text, f
        assert "python bench.py" in text, f


L2_BYTES = 135_475_200   # the L2 size the GB300 reports (torch device properties), as in bench.py's line


def _fields(name):
    out = {}
    for line in open(os.path.join(PROFILES, name)):
        line = line.lstrip("# ").strip()
        for key in ("algorithmic_read_bytes", "algorithmic_write_bytes", "dram_read_bytes", "dram_write_bytes",
                    "traffic_bytes_per_launch"):
            if line.startswith(key + ":"):
                v = line.split(":", 1)[1].split()
                if v and v[0].replace(".", "", 1).isdigit():
                    out[key] = float(v[0])
    return out


def test_captured_dram_bytes_match_algorithmic_bytes():
    """Every summary that records a DRAM capture: reads within 5 % of the algorithmic reads;
    writes within 5 % above the algorithmic writes and at most one L2 below them (output still
    dirty in L2 when the kernel ends is written back after it); traffic = reads + writes."""
    seen = 0
    for f in sorted(os.listdir(PROFILES)):
        d = _fields(f)
        if "dram_read_bytes" not in d:
            continue
        seen += 1
        r, ar = d["dram_read_bytes"], d["algorithmic_read_bytes"]
        assert 0.95 * ar <= r <= 1.05 * ar, (f, r, ar)
        if "algorithmic_write_bytes" in d and d["algorithmic_write_bytes"] > 1e6:
            w, aw = d["dram_write_bytes"], d["algorithmic_write_bytes"]
            assert aw - L2_BYTES <= w <= 1.05 * aw + 8e6, (f, w, aw)
        assert d["traffic_bytes_per_launch"] == d["dram_read_bytes"] + d["dram_write_bytes"], f
    assert seen >= 4
