"""GPU parity of lla_backward against the fp64 oracle's backward.

Small and ragged shapes are compared element by element with the full oracle
backward (all five gradients); the headline-size problem is compared on sampled
positions computed one by one by the oracle (dq, dk, dv, dlambda rows, and the
differences dlog_a_x - dlog_a_{x+1}).
"""
import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import rel_err_per_head, to_device, torch_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def _dout(cfg, B, H, T, seed):
    g = np.random.default_rng(seed).normal(size=(B, H, T, cfg.dv))
    if cfg.dtype == "bf16":
        bits = inputs.f32_to_bf16_bits(g.astype(np.float32))
        return inputs.bf16_bits_to_f32(bits).astype(np.float64), torch_bf16(bits, "cuda")
    g32 = g.astype(np.float32)
    return g32.astype(np.float64), torch.from_numpy(g32).cuda()


def _run(cfg, seed, chunk):
    from log_linear_attention_gb300 import binding
    inp = inputs.make_prefill(cfg, seed=seed)
    q, k, v, log_a, lam = to_device(inp)
    g_host, g_dev = _dout(cfg, cfg.B, cfg.H, cfg.T, seed + 1000)
    grads = binding.backward(q, k, v, log_a, lam, g_dev, chunk)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return inp, g_host, [x.float().cpu().numpy().astype(np.float64) for x in grads]


@pytest.mark.parametrize("B,H,T,dk,dv,chunk,dtype", [
    (1, 1, 16, 16, 16, 16, "f32"),
    (2, 2, 64, 8, 4, 16, "f32"),
    (1, 2, 96, 24, 40, 32, "f32"),
    (1, 1, 256, 16, 16, 64, "f32"),
    (2, 1, 384, 64, 32, 128, "f32"),
    (1, 2, 256, 64, 64, 64, "bf16"),      # dk != 128: CUDA-core kernels
    (1, 1, 640, 128, 128, 128, "bf16"),   # dv = 128: CUDA-core kernels
    # bf16, dk = 128, dv = 64, T % 128 == 0: tensor-core kernels
    (1, 1, 128, 128, 64, 64, "bf16"),     # one tile, no node
    (1, 2, 384, 128, 64, 64, "bf16"),
    (2, 2, 512, 128, 64, 64, "bf16"),
    (2, 1, 1024, 128, 64, 128, "bf16"),
    (1, 1, 2304, 128, 64, 64, "bf16"),    # 18 tiles
    (1, 9, 2176, 128, 64, 64, "bf16"),    # 153 (head, tile) items: one more than a GB300 has SMs
])
def test_backward_matches_oracle(B, H, T, dk, dv, chunk, dtype):
    cfg = inputs.PrefillConfig("bw", B, H, T, dk, dv, chunk, dtype)
    inp, g, got = _run(cfg, seed=T + dk + dv, chunk=chunk)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.log_a, inp.lam, g)
    tol = 1e-4 if dtype == "f32" else 2e-2
    names = ["dq", "dk", "dv", "dlog_a", "dlambda"]
    for name, a, r in zip(names, got, ref):
        if name == "dlog_a":
            a, r = a[..., None], r[..., None]
        err = rel_err_per_head(a, r)
        assert err <= tol, (name, err)


@pytest.mark.parametrize("mu", [2.0, 4.0])
def test_backward_fast_decay(mu):
    """Strong decays on the tensor-core path: at mu = 4 every 32-token block decays by more
    than 100 bits, so the diagonal blocks of the tile kernel take their exact per-key decay;
    at mu = 2 most blocks take the factorised one and some do not."""
    cfg = inputs.PrefillConfig("bwfast", 1, 2, 512, 128, 64, 64, "bf16", log_a_mu=mu)
    inp, g, got = _run(cfg, seed=21, chunk=64)
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.log_a, inp.lam, g)
    for name, a, r in zip(["dq", "dk", "dv", "dlog_a", "dlambda"], got, ref):
        if name == "dlog_a":
            a, r = a[..., None], r[..., None]
        err = rel_err_per_head(a, r)
        assert err <= 2e-2, (name, err)


def test_backward_chunk_invariance():
    cfg = inputs.PrefillConfig("bwc", 1, 2, 512, 32, 32, 16, "f32")
    outs = [_run(cfg, seed=3, chunk=c)[2] for c in (16, 32, 64)]
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            if a.ndim == 3:
                a, b = a[..., None], b[..., None]
            assert rel_err_per_head(b, a) <= 1e-4


def test_backward_headline_sampled():
    """4 x 16 heads x 8192 tokens, bf16, dk 128, dv 64: sampled positions of two heads."""
    cfg = inputs.PREFILL_CONFIGS["headline"]
    inp, g, (dq, dk, dv, dla, dlam) = _run(cfg, seed=0, chunk=cfg.chunk)
    rows = [0, 1, 63, 64, 127, 128, 2047, 4095, 4096, 6000, 8190, 8191]
    for b, h in ((0, 3), (3, 14)):
        rq, rk, rv, rl, rc = oracle.backward_rows(inp.q, inp.k, inp.v, inp.log_a, inp.lam, g, b, h, rows)
        nxt = np.append(dla[b, h], 0.0)
        gc = nxt[rows] - nxt[np.array(rows) + 1]
        for name, a, r in (("dq", dq[b, h, rows], rq), ("dk", dk[b, h, rows], rk), ("dv", dv[b, h, rows], rv),
                           ("dlambda", dlam[b, h, rows], rl)):
            err = np.abs(a - r).max() / np.abs(r).max()
            assert err <= 2e-2, (name, (b, h), err)
        # dcum from differences of a running sum: compare against the scale of dlog_a itself
        err = np.abs(gc - rc).max() / max(np.abs(rc).max(), 1e-30)
        assert err <= 2e-2, ("dcum", (b, h), err)


def test_backward_long_sampled():
    """1 x 2 heads x 65536 tokens, bf16, dk 128, dv 64: 512 tiles, nine node levels, so the
    node-gradient kernel runs a second level window (level 8). Sampled positions of both heads,
    including the block boundaries of the top levels."""
    cfg = inputs.PrefillConfig("bwlong", 1, 2, 65536, 128, 64, 128, "bf16", qk_unit_rows=True, log_a_mu=-2.0)
    inp, g, (dq, dk, dv, dla, dlam) = _run(cfg, seed=5, chunk=cfg.chunk)
    rows = [0, 127, 128, 255, 256, 32767, 32768, 32895, 40000, 49152, 65407, 65535]
    for b, h in ((0, 0), (0, 1)):
        rq, rk, rv, rl, rc = oracle.backward_rows(inp.q, inp.k, inp.v, inp.log_a, inp.lam, g, b, h, rows)
        nxt = np.append(dla[b, h], 0.0)
        gc = nxt[rows] - nxt[np.array(rows) + 1]
        for name, a, r in (("dq", dq[b, h, rows], rq), ("dk", dk[b, h, rows], rk), ("dv", dv[b, h, rows], rv),
                           ("dlambda", dlam[b, h, rows], rl)):
            err = np.abs(a - r).max() / np.abs(r).max()
            assert err <= 2e-2, (name, (b, h), err)
        err = np.abs(gc - rc).max() / max(np.abs(rc).max(), 1e-30)
        assert err <= 2e-2, ("dcum", (b, h), err)
