"""Layer shapes beyond the workloads, against the oracle: the largest E the
library takes (1024, with enough tiles for the round-robin whole-tile
schedule), every expert selected (k = E = 64), odd tile and chunk counts
(H = 384: three 128-row tiles of the down GEMM and three K chunks of the
gate+up GEMM; I = 128: one K chunk of the down GEMM), the 128-row token
tile of the down GEMM, which the library only picks when told to, and the
CTA-pair kernels (128- and 160-row gate+up and 64-row down token tiles) on
experts of every ragged row count, next to a down GEMM whose odd number of
weight tiles keeps it on single CTAs."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(L, M, seed=0):
    """The whole batch: every token's output and every slot's act and y."""
    import quantized_moe_expert_align_gb300 as moe
    dl = gu.DeviceLayer(L, seed)
    x = synth.hidden(M, L.H, seed)
    ids, w = synth.routing(M, L, seed)
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    what = f"E{L.E} H{L.H} I{L.I} k{L.k} M{M}"
    ref, _ = gu.check_stages(dl, x, ids, w, ws.buf, np.arange(M * L.k), what)
    return gu.parity(gu.bf16_dev_to_f64(out), ref["out"], what)


def _run_counts(L, counts, seed=0):
    """k = 1, expert e routed exactly counts[e] tokens (in a shuffled order),
    all routing weights 1; every token's output and every slot's act and y."""
    import quantized_moe_expert_align_gb300 as moe
    rng = np.random.default_rng(seed)
    ids = np.repeat(np.arange(L.E, dtype=np.int32), counts)
    ids = ids[rng.permutation(ids.size)].reshape(-1, 1)
    M = ids.shape[0]
    w = np.ones((M, 1), np.float32)
    dl = gu.DeviceLayer(L, seed)
    x = synth.hidden(M, L.H, seed)
    out, ws = dl.forward(x, ids, w)
    st, _ = moe.moe_w4a16_get_device_status(ws.buf)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    what = f"E{L.E} H{L.H} I{L.I} counts {list(counts)}"
    ref, _ = gu.check_stages(dl, x, ids, w, ws.buf, np.arange(M), what)
    gu.parity(gu.bf16_dev_to_f64(out), ref["out"], what)
    return moe.moe_w4a16_get_diag()["token_tile"]


# rows per expert around every multiple of 16 and 32 up to two 128-row tiles
_RAGGED = [1, 15, 16, 17, 31, 33, 47, 48, 63, 64, 65, 95, 97, 127, 128, 129, 160, 200, 255, 256]


def test_cta_pairs_ragged_tiles(gpu):
    """Both GEMMs on CTA pairs (4 and 2 weight tiles per expert): gate+up
    token tiles whose rows round up to 32, 64, 96 or 128 MMA columns (half
    of them in each CTA), down tiles of 1-64 rows."""
    assert _run_counts(synth.Layer(20, 256, 256, 1), _RAGGED) == 128


def test_cta_pairs_next_to_single_ctas(gpu):
    """H = 384: the down GEMM's three weight tiles per expert keep it on
    single CTAs (64-row token tiles) while the gate+up GEMM runs on pairs."""
    assert _run_counts(synth.Layer(20, 384, 128, 1), _RAGGED[::-1], seed=1) == 128


# rows per expert around every multiple of 32 up to two 160-row tiles, with
# enough rows on average (about 128) for 160-row gate+up tiles
_RAGGED_160 = [1, 31, 33, 95, 97, 127, 128, 129, 140, 152, 159, 160, 161, 175, 190, 200,
               250, 300, 319, 320]


def test_cta_pairs_160_row_tiles(gpu):
    """160-row gate+up tiles (80 rows in each CTA of a pair, MMAs of 32-160
    columns) and 64-row down tiles."""
    assert _run_counts(synth.Layer(20, 256, 256, 1), _RAGGED_160, seed=2) == 160


def test_eight_row_tiles_with_a_heavy_expert(gpu):
    """A decode-sized batch (at least 32 slots, at most 3 rows per active
    expert) runs both GEMMs on 8-row token tiles; one expert spans five of
    them, the last ragged.  Every token's output and every slot's act and y."""
    import quantized_moe_expert_align_gb300 as moe
    assert _run_counts(synth.Layer(32, 256, 256, 1), [37] + [1] * 31, seed=3) == 8
    assert moe.moe_w4a16_get_diag()["token_tile2"] == 8


def test_e1024_round_robin(gpu):
    import quantized_moe_expert_align_gb300 as moe
    L = synth.Layer(1024, 256, 128, 8)
    _run(L, 2048)
    assert moe.moe_w4a16_get_diag()["token_tile"] == 32


def test_every_expert_selected(gpu):
    _run(synth.Layer(64, 256, 128, 64), 24)


@pytest.mark.parametrize("M", [3, 200])
def test_odd_tiles_and_chunks(gpu, M):
    _run(synth.Layer(16, 384, 128, 4), M)


_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import synth
from tests import gpu_util as gu
import quantized_moe_expert_align_gb300 as moe
L = synth.Layer(32, 256, 256, 8)
M = 600
dl = gu.DeviceLayer(L, 0)
x = synth.hidden(M, L.H, 0)
ids, w = synth.routing(M, L, 0)
out, ws = dl.forward(x, ids, w)
st, _ = moe.moe_w4a16_get_device_status(ws.buf)
ratio, rel = gu.parity(gu.bf16_dev_to_f64(out), dl.oracle(x, ids, w), "forced 128")
print(json.dumps({"status": st, "tile": moe.moe_w4a16_get_diag()["token_tile"],
                  "ratio": ratio, "rel": rel}))
"""


def test_forced_128_row_tiles(gpu):
    """Both GEMMs on 128-row token tiles (the down GEMM's separate hi and lo
    MMAs); the tile choice is read once per process, so in a child."""
    env = dict(os.environ, MOE_W4A16_TOKEN_TILE="128")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == 0 and res["tile"] == 128
