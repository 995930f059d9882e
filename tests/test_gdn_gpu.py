"""GPU parity of the log-linear Gated DeltaNet (lla_gdn_forward, lla_gdn_decode_step) against
the fp64 CPU oracle on the same seeded inputs.

Metric as everywhere: max over heads of ||o_gpu - o_ref||_inf / ||o_ref||_inf; 1e-4 for fp32
inputs, 2e-2 for bf16 inputs (all GPU arithmetic here is fp32; bf16 only in storage).
"""
import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import decode_to_device, rel_err_per_head, to_device, torch_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def _cfg(name, **over):
    base = inputs.GDN_CONFIGS.get(name) or inputs.PREFILL_CONFIGS[name]
    d = dict(base.__dict__)
    d.update(over)
    d.setdefault("qk_unit_rows", True)
    d["qk_unit_rows"] = True
    return inputs.PrefillConfig(**d)


def _problem(cfg, seed):
    inp = inputs.make_prefill(cfg, seed=seed)
    beta = inputs.make_beta(seed, (cfg.B, cfg.H, cfg.T))
    return inp, beta


def _run(inp, beta, chunk):
    from log_linear_attention_gb300 import binding
    q, k, v, log_a, lam = to_device(inp)
    out = binding.gdn_forward(q, k, v, log_a, torch.from_numpy(beta).cuda(), lam, chunk)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return out.float().cpu().numpy()


def _ref(inp, beta):
    args = (inp.q, inp.k, inp.v, inp.log_a, beta, inp.lam)
    return oracle.gdn_explicit(*args) if inp.cfg.T <= 256 else oracle.gdn_recurrent(*args)


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_gdn_oracle_scale_fp32(chunk):
    cfg = _cfg("gdn-oracle-scale")
    inp, beta = _problem(cfg, 1)
    assert rel_err_per_head(_run(inp, beta, chunk), _ref(inp, beta)) <= TOL_F32


@pytest.mark.parametrize("B,H,T,dk,dv,chunk", [
    (2, 3, 192, 24, 32, 64),    # 3 chunks (not a power of two), odd dk
    (1, 2, 192, 24, 16, 16),    # 12 chunks
    (1, 1, 16, 16, 16, 16),     # a single chunk: no inter-chunk level
    (1, 1, 48, 1, 16, 16),      # dk = 1
    (1, 1, 256, 128, 128, 128), # largest head sizes, chunk 128 run as 64
])
def test_gdn_fp32_ragged_shapes(B, H, T, dk, dv, chunk):
    cfg = _cfg("gdn-oracle-scale", B=B, H=H, T=T, dk=dk, dv=dv, chunk=chunk)
    inp, beta = _problem(cfg, T + dk)
    assert rel_err_per_head(_run(inp, beta, chunk), _ref(inp, beta)) <= TOL_F32


@pytest.mark.parametrize("T,dk,dv,chunk", [(128, 128, 64, 64), (1024, 128, 64, 64), (640, 128, 64, 64),
                                            (512, 64, 64, 32), (2048, 64, 128, 64)])
def test_gdn_bf16_shapes(T, dk, dv, chunk):
    cfg = _cfg("gdn-headline", B=1, H=2, T=T, dk=dk, dv=dv, chunk=chunk)
    inp, beta = _problem(cfg, T + dv)
    assert rel_err_per_head(_run(inp, beta, chunk), _ref(inp, beta)) <= TOL_BF16


@pytest.mark.parametrize("dk", [128, 64])
def test_gdn_bf16_levels_run_on_tensor_cores(dk):
    """bf16 with chunk 64 and dv = 64 runs the chunk pass and the Fenwick level carries on
    tcgen05 (gdn_chunk_tc, gdn_level_tc), at dk = 128 and at dk = 64 (zero-padded operands);
    the result matches the oracle."""
    from log_linear_attention_gb300 import binding
    cfg = _cfg("gdn-headline", B=1, H=2, T=1024, dk=dk)
    inp, beta = _problem(cfg, 40 + dk)
    q, k, v, log_a, lam = to_device(inp)
    out = torch.empty_like(v)
    names = [n for n, _ in binding.gdn_forward_profile(q, k, v, log_a, torch.from_numpy(beta).cuda(), lam, 64, out)]
    assert binding.device_error() == 0
    assert names[0] == "gdn_chunk_tc" and "gdn_level_tc" in names and "gdn_level" not in names, names
    assert rel_err_per_head(out.float().cpu().numpy(), _ref(inp, beta)) <= TOL_BF16


@pytest.mark.parametrize("B,H,T,dk", [(2, 3, 64, 128), (1, 2, 64, 64), (3, 1, 128, 64)])
def test_gdn_tensor_core_short_sequences(B, H, T, dk):
    """The tensor-core chunk pass on one chunk (its output goes straight to `out`, no level pass)
    and on two chunks (one level-0 read), at dk = 128 and 64."""
    from log_linear_attention_gb300 import binding
    cfg = _cfg("gdn-headline", B=B, H=H, T=T, dk=dk)
    inp, beta = _problem(cfg, 60 + T + dk)
    q, k, v, log_a, lam = to_device(inp)
    out = torch.empty_like(v)
    names = [n for n, _ in binding.gdn_forward_profile(q, k, v, log_a, torch.from_numpy(beta).cuda(), lam, 64, out)]
    assert binding.device_error() == 0
    assert names[0] == "gdn_chunk_tc", names
    assert rel_err_per_head(out.float().cpu().numpy(), _ref(inp, beta)) <= TOL_BF16


def test_gdn_slow_decay_long_range():
    """log_a near 0 keeps far keys alive, so the coarse Fenwick levels (and the carried
    transitions through many chunks) carry much of the output."""
    cfg = _cfg("gdn-headline", B=1, H=2, T=4096, log_a_mu=-9.0)
    inp, beta = _problem(cfg, 5)
    assert rel_err_per_head(_run(inp, beta, 64), _ref(inp, beta)) <= TOL_BF16


def test_gdn_chunk_invariance():
    cfg = _cfg("gdn-small", B=1, H=2, T=1024)
    inp, beta = _problem(cfg, 3)
    outs = [_run(inp, beta, c) for c in (16, 32, 64)]
    ref = _ref(inp, beta)
    for o in outs:
        assert rel_err_per_head(o, ref) <= TOL_BF16


def test_gdn_full_size_sampled_rows():
    """The full headline-shaped workload (B4 H16 T8192 dk128 dv64, bf16) in the benchmark's launch
    configuration; the oracle computes sampled rows of three heads one by one."""
    cfg = inputs.GDN_CONFIGS["gdn-headline"]
    inp, beta = _problem(cfg, 0)
    got = _run(inp, beta, cfg.chunk)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(7)
    for b, h in [(0, 0), (cfg.B - 1, cfg.H - 1), (cfg.B // 2, cfg.H // 3)]:
        rows = sorted({0, 1, 63, 64, 65, 127, 128, 4095, 4096, cfg.T - 2, cfg.T - 1}
                      | {int(x) for x in rng.integers(0, cfg.T, 12)})
        ref = oracle.gdn_explicit_rows(inp.q, inp.k, inp.v, inp.log_a, beta, inp.lam, b, h, rows)
        err = np.abs(got[b, h, rows] - ref).max() / np.abs(ref).max()
        assert err <= TOL_BF16, (b, h, err)


# ---------------------------------------------------------------- decode


def _decode_case(dtype, batch, H, dk, dv, t_max, seed):
    dcfg = inputs.DecodeConfig("gdn-decode", batch=batch, H=H, dk=dk, dv=dv, t_max=t_max, steps=1, Lmax=18,
                               dtype=dtype)
    tok = inputs.make_decode_token(dcfg, seed)
    # unit-norm keys, as the prefill workloads use
    k = tok.k / np.linalg.norm(tok.k, axis=-1, keepdims=True)
    if dtype == "bf16":
        kb = inputs.f32_to_bf16_bits(k)
        tok.bits["k"] = kb
        k = inputs.bf16_bits_to_f32(kb).reshape(k.shape)
    tok.k = k
    beta = inputs.make_beta(seed, (batch, H))
    states = inputs.make_random_states(dcfg, seed)
    pos = inputs.make_positions(dcfg, seed)
    return dcfg, tok, beta, states, pos


@pytest.mark.parametrize("dtype,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 64), (16, 16), (32, 128), (128, 128)])
def test_gdn_decode_random_states(dtype, tol, dk, dv):
    from log_linear_attention_gb300 import binding
    dcfg, tok, beta, st0, pos = _decode_case(dtype, 6, 3, dk, dv, 5000, dk + dv)
    states = torch.from_numpy(st0).cuda()
    q, k, v, log_a, lam = decode_to_device(tok, dtype)
    out = binding.gdn_decode_step(q, k, v, log_a, torch.from_numpy(beta).cuda(), lam, states,
                                  torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref_states = st0.astype(np.float64)
    ref = oracle.gdn_decode_step(tok.q, tok.k, tok.v, tok.log_a, beta, tok.lam, ref_states, pos)
    assert rel_err_per_head(out.float().cpu().numpy()[..., None, :], ref[..., None, :]) <= tol
    # every slot the step wrote: the merged level, the carried coarser levels and level 0
    got = states.cpu().numpy()
    for b, t in enumerate(pos.tolist()):
        held = [0] + [l for l in range(1, dcfg.Lmax) if (t >> (l - 1)) & 1]
        for l in held:
            err = np.abs(got[b, :, l] - ref_states[b, :, l]).max() / np.abs(ref_states[b, :, l]).max()
            assert err <= 1e-4, (b, t, l, err)


def test_gdn_decode_from_empty_matches_forward():
    """Stepping the decode kernel from empty states over a sequence reproduces the prefill's
    rows (two GPU paths of the same operator), and both match the oracle."""
    from log_linear_attention_gb300 import binding
    cfg = _cfg("gdn-oracle-scale", B=2, H=2, T=96, dk=32, dv=16, chunk=32)
    inp, beta = _problem(cfg, 21)
    fwd = _run(inp, beta, cfg.chunk)
    q, k, v, log_a, lam = to_device(inp)
    bt = torch.from_numpy(beta).cuda()
    Lmax = inputs.num_levels(cfg.T)
    states = torch.zeros((cfg.B, cfg.H, Lmax, cfg.dk, cfg.dv), dtype=torch.float32, device="cuda")
    rows = []
    for t in range(cfg.T):
        pos = torch.full((cfg.B,), t, dtype=torch.int64, device="cuda")
        o = binding.gdn_decode_step(q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(),
                                    log_a[:, :, t].contiguous(), bt[:, :, t].contiguous(),
                                    lam[:, :, t].contiguous(), states, pos)
        rows.append(o.float().cpu().numpy())
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    dec = np.stack(rows, axis=2)
    assert rel_err_per_head(dec, fwd) <= TOL_F32
    assert rel_err_per_head(dec, _ref(inp, beta)) <= TOL_F32


def test_gdn_decode_rejects_out_of_range_position():
    from log_linear_attention_gb300 import binding
    dcfg, tok, beta, st0, pos = _decode_case("f32", 2, 1, 16, 16, 100, 3)
    pos[1] = 1 << 20  # needs 22 levels; the state set holds 18
    states = torch.from_numpy(st0).cuda()
    before = states[1].clone()
    q, k, v, log_a, lam = decode_to_device(tok, "f32")
    binding.gdn_decode_step(q, k, v, log_a, torch.from_numpy(beta).cuda(), lam, states, torch.from_numpy(pos).cuda())
    assert binding.device_error() == binding.LLA_ERR_DEVICE
    assert torch.equal(states[1], before)
