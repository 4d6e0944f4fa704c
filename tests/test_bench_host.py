"""bench.py's reference arm on the CPU (no GPU): it prints one JSON line
with the keys the bench contract asks for, for a layer workload and for
the GPTQ repack configuration."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "config", "cpu_baseline", "e2e")


@pytest.mark.parametrize("config", ["tiny", "gptq_repack"])
def test_reference_arm_prints_one_json_line(config):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", config, "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_path_choice_mirrors_the_header():
    """bench.py labels a workload decode or GEMM by the same token count at
    which QMOE_PATH_AUTO switches (include/qmoe.h), so its per-kernel names
    and byte counts follow the path the library runs."""
    import re
    sys.path.insert(0, ROOT)
    from int4_block_quantized_gb300 import binding, synthetic as S
    import bench
    hdr = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    auto = int(re.search(r"#define QMOE_AUTO_DECODE_MAX_TOKENS (\d+)", hdr).group(1))
    top = int(re.search(r"#define QMOE_DECODE_MAX_TOKENS (\d+)", hdr).group(1))
    assert binding.AUTO_DECODE_MAX_TOKENS == auto and binding.DECODE_MAX_TOKENS == top
    base = S.WORKLOADS["verify"]
    for T in (1, auto, auto + 1, 16, 512):
        wl = S.Workload("t%d" % T, T, base.H, base.I, base.E, base.k, base.block_size, base.act_dtype,
                        base.scale_dtype, base.has_zp, base.scale_exp)
        assert bench.is_decode(wl) == (T <= auto)


def test_tile_columns_helper_matches_a_direct_split():
    """tests/qmoe_check.tile_columns (which the full-size GPU parity tests
    use to pick tokens covering every token-tile column) against a direct
    simulation of the grouping and the tile split."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from qmoe_check import tile_columns, tokens_covering_tile_columns
    rng = np.random.default_rng(0)
    for T, E, k, tile in ((2048, 60, 4, 160), (512, 8, 2, 160), (300, 2, 1, 160)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
        cols = tile_columns(ids, E, tile).reshape(-1)
        flat = ids.reshape(-1)
        for e in range(E):
            a = np.nonzero(flat == e)[0]
            n = a.size
            if n == 0:
                continue
            nt = 1 if n <= tile else -(-n // 128)
            rows = -(-n // nt)
            assert rows <= tile
            assert (cols[a] == np.arange(n) % rows).all()
        picked = tokens_covering_tile_columns(ids, E, 16, 1, tile)
        assert set(np.unique(tile_columns(ids, E, tile)[picked])) == set(np.unique(cols))
