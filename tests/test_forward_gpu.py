"""GPU parity of lla_forward against the fp64 CPU oracle on the same seeded inputs.

Metric: max over heads of ||o_gpu - o_ref||_inf / ||o_ref||_inf. Bars: 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs (bf16 output rounding alone is 2^-9; bf16
operands of the tensor-core products add a few 2^-9 more).
"""
import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import rel_err_per_head, to_device

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()  # fails loudly if the library was not built


def run(inp, chunk, **kw):
    from log_linear_attention_gb300 import binding
    q, k, v, log_a, lam = to_device(inp)
    out = binding.forward(q, k, v, log_a, lam, chunk, **kw)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return out.float().cpu().numpy()


def oracle_full(inp):
    if inp.cfg.T <= 256:
        return oracle.explicit(inp.q, inp.k, inp.v, inp.log_a, inp.lam)
    return oracle.recurrent(inp.q, inp.k, inp.v, inp.log_a, inp.lam)


def cfg_like(name, **over):
    c = inputs.PREFILL_CONFIGS[name]
    d = dict(c.__dict__)
    d.update(over)
    return inputs.PrefillConfig(**d)


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_oracle_scale_fp32(chunk):
    cfg = inputs.PREFILL_CONFIGS["oracle-scale"]
    inp = inputs.make_prefill(cfg, seed=1)
    got = run(inp, chunk)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_F32


@pytest.mark.parametrize("B,H,T,dk,dv,chunk", [
    (2, 3, 192, 24, 40, 64),   # N = 3 chunks (not a power of two), odd head sizes
    (1, 2, 192, 24, 40, 16),   # N = 12
    (1, 1, 16, 16, 16, 16),    # a single chunk: no inter-chunk level
    (3, 1, 128, 128, 128, 32), # largest head sizes on the fp32 path
    (1, 1, 48, 1, 4, 16),      # dk = 1
])
def test_fp32_ragged_shapes(B, H, T, dk, dv, chunk):
    cfg = cfg_like("oracle-scale", B=B, H=H, T=T, dk=dk, dv=dv, chunk=chunk)
    inp = inputs.make_prefill(cfg, seed=T + dk)
    got = run(inp, chunk)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_F32


def test_small_bf16():
    cfg = inputs.PREFILL_CONFIGS["small"]
    inp = inputs.make_prefill(cfg, seed=2)
    got = run(inp, cfg.chunk)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_BF16


def test_small_bf16_runs_on_tensor_cores():
    """dk = dv = 64 in bf16 takes the tcgen05 kernels (q and k zero-padded to 128 columns by
    TMA), not the fp32 CUDA-core kernels."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PREFILL_CONFIGS["small"]
    inp = inputs.make_prefill(cfg, seed=2)
    q, k, v, log_a, lam = to_device(inp)
    names = [n for n, _ in binding.forward_profile(q, k, v, log_a, lam, cfg.chunk, torch.empty_like(v))]
    assert names == ["tc_nodes", "tc_merge", "tc_output"], names


@pytest.mark.parametrize("T,dv", [(256, 64), (1152, 128)])
def test_bf16_dk64_shapes(T, dv):
    """dk = 64 on the tensor-core path at dv = 64 and 128, several tiles and a tile count
    that is not a power of two."""
    cfg = cfg_like("small", B=2, H=1, T=T, dv=dv, chunk=64)
    inp = inputs.make_prefill(cfg, seed=T + 17)
    got = run(inp, 64)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_BF16


@pytest.mark.parametrize("T,dv,chunk", [(128, 64, 64), (1024, 64, 64), (640, 64, 128), (2048, 128, 128),
                                        (384, 64, 32)])
def test_bf16_dk128_shapes(T, dv, chunk):
    """dk = 128 bf16 shapes (the tensor-core path): several 128-token tiles, a
    non-power-of-two tile count, dv = 64 and 128."""
    cfg = cfg_like("headline", B=1, H=2, T=T, dv=dv, chunk=chunk)
    inp = inputs.make_prefill(cfg, seed=T + dv)
    got = run(inp, chunk)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_BF16


def test_bf16_slow_decay_long_range():
    """log_a near 0 keeps far keys alive, so the coarse Fenwick levels carry most of the output."""
    cfg = cfg_like("headline", B=1, H=2, T=4096, log_a_mu=-9.0)
    inp = inputs.make_prefill(cfg, seed=5)
    got = run(inp, 64)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_BF16


@pytest.mark.parametrize("mu", [2.0, 4.0])
def test_bf16_fast_decay(mu):
    """Strong decays: at mu = 4 every 32-token block decays by more than 100 bits, so the
    diagonal blocks of the tensor-core output kernel take their exact per-key decay; at
    mu = 2 (about 95 bits a block) most blocks take the factorised one and some do not."""
    cfg = cfg_like("headline", B=1, H=2, T=512, log_a_mu=mu)
    inp = inputs.make_prefill(cfg, seed=11)
    got = run(inp, 64)
    assert rel_err_per_head(got, oracle_full(inp)) <= TOL_BF16


def test_chunk_invariance_bf16():
    cfg = cfg_like("small", B=1, H=2, T=1024)
    inp = inputs.make_prefill(cfg, seed=3)
    outs = [run(inp, c) for c in (16, 32, 64, 128)]
    ref = oracle_full(inp)
    for o in outs:
        assert rel_err_per_head(o, ref) <= TOL_BF16
        assert rel_err_per_head(o, outs[-1]) <= TOL_BF16


def test_caller_workspace_matches_pool_workspace():
    from log_linear_attention_gb300 import binding
    cfg = cfg_like("headline", B=1, H=2, T=1024)
    inp = inputs.make_prefill(cfg, seed=4)
    q, k, v, log_a, lam = to_device(inp)
    nbytes = binding.workspace_size(1, 2, 1024, 128, 64, 64, torch.bfloat16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    a = binding.forward(q, k, v, log_a, lam, 64)
    b = binding.forward(q, k, v, log_a, lam, 64, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_host_buffers_end_to_end():
    """CPU tensors in, CPU tensor out: the binding stages the copies around the same call."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PREFILL_CONFIGS["oracle-scale"]
    inp = inputs.make_prefill(cfg, seed=6)
    q, k, v, log_a, lam = (t.cpu() for t in to_device(inp))
    out = binding.forward(q, k, v, log_a, lam, 16)
    assert out.device.type == "cpu"
    assert rel_err_per_head(out.numpy(), oracle_full(inp)) <= TOL_F32


def _sampled_rows(T, tile, rng, n_random=24):
    rows = {0, 1, T - 1, T - 2}
    for base in (tile, 2 * tile, T // 2, T - tile):
        rows.update({base - 1, base, base + 1})
    rows.update(int(x) for x in rng.integers(0, T, n_random))
    return sorted(r for r in rows if 0 <= r < T)


@pytest.mark.parametrize("name", ["headline", "long"])
def test_full_size_sampled_rows(name):
    """Full benchmark sizes in the benchmark's launch configuration; the oracle computes
    sampled rows of a few heads one by one (explicit form)."""
    cfg = inputs.PREFILL_CONFIGS[name]
    inp = inputs.make_prefill(cfg, seed=0)
    got = run(inp, cfg.chunk)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(7)
    heads = [(0, 0), (cfg.B - 1, cfg.H - 1), (cfg.B // 2, cfg.H // 3)]
    for b, h in heads:
        rows = _sampled_rows(cfg.T, 128, rng)
        ref = oracle.explicit_rows(inp.q, inp.k, inp.v, inp.log_a, inp.lam, b, h, rows)
        err = np.abs(got[b, h, rows] - ref).max() / np.abs(ref).max()
        assert err <= TOL_BF16, (b, h, err)


@pytest.mark.parametrize("B,H,T,dk,dv,dtype,chunk", [(1, 5, 256, 128, 64, "bf16", 64), (2, 3, 96, 16, 24, "f32", 32)])
def test_host_buffers_match_device_path(B, H, T, dk, dv, dtype, chunk):
    """lla_forward_host (head groups copied in, run and copied out on separate streams) gives
    the device path's result exactly, from pageable inputs into a pinned output."""
    from log_linear_attention_gb300 import binding
    cfg = inputs.PrefillConfig("host", B, H, T, dk, dv, chunk, dtype)
    inp = inputs.make_prefill(cfg, seed=5)
    dev = to_device(inp)
    ref = binding.forward(*dev, chunk).cpu()
    host = [x.cpu() for x in dev]
    out = torch.empty(ref.shape, dtype=ref.dtype, pin_memory=True)
    got = binding.forward(*host, chunk, out=out)
    assert got.data_ptr() == out.data_ptr()
    assert torch.equal(got, ref)
    with pytest.raises(binding.LLAError):
        binding.load()
        st = binding.load().lla_forward_host(dev[0].data_ptr(), host[1].data_ptr(), host[2].data_ptr(),
                                             host[3].data_ptr(), host[4].data_ptr(), out.data_ptr(), B, H, T, dk, dv,
                                             chunk, None, binding.LLA_BF16 if dtype == "bf16" else binding.LLA_F32)
        binding._call(st, "lla_forward_host")
