"""GPU checks of the packed variable-length entry points against the oracle, sequence by
sequence: lla_forward_varlen outputs, lla_prefill_state_varlen states, decode steps that
continue each sequence from its own position, and a malformed cu_seqlens."""
import types

import numpy as np
import pytest

import oracle
from log_linear_attention_gb300 import inputs
from tests._util import rel_err_per_head, torch_bf16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from log_linear_attention_gb300 import binding
    binding.load()


def packed_problem(lengths, H, dk, dv, dtype, seed):
    """Per-sequence problems (each its own positions 0..len-1) and their packed concatenation."""
    max_T = max(lengths)
    L = inputs.num_levels(max_T)
    seqs = []
    for b, n in enumerate(lengths):
        cfg = inputs.PrefillConfig("vl", 1, H, n, dk, dv, 16, dtype)
        seqs.append(inputs.make_prefill(cfg, seed=seed + b))
    rng = np.random.default_rng(seed + 999)

    def cat(name):
        return np.concatenate([getattr(x, name)[0] for x in seqs], axis=1)

    lam = np.concatenate([np.concatenate([x.lam[0], np.log1p(np.exp(rng.normal(size=(H, x.lam.shape[2], L - x.lam.shape[3]))))], axis=-1)
                          for x in seqs], axis=1)
    packed = types.SimpleNamespace(q=cat("q"), k=cat("k"), v=cat("v"), log_a=cat("log_a"), lam=lam)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return seqs, packed, cu, max_T


def to_dev(packed, seqs, dtype):
    if dtype == "bf16":
        bits = {n: np.concatenate([x.bits[n][0] for x in seqs], axis=1) for n in ("q", "k", "v")}
        q, k, v = (torch_bf16(bits[n], "cuda") for n in ("q", "k", "v"))
    else:
        q, k, v = (torch.from_numpy(np.ascontiguousarray(getattr(packed, n), dtype=np.float32)).cuda()
                   for n in ("q", "k", "v"))
    la = torch.from_numpy(np.ascontiguousarray(packed.log_a, dtype=np.float32)).cuda()
    lam = torch.from_numpy(np.ascontiguousarray(packed.lam, dtype=np.float32)).cuda()
    return q, k, v, la, lam


@pytest.mark.parametrize("lengths,H,dk,dv,chunk,dtype", [
    ([1, 37, 128, 300, 16], 2, 16, 16, 16, "f32"),
    ([64, 5, 200], 1, 24, 40, 32, "f32"),
    ([100, 640, 257, 1024, 1], 2, 128, 64, 64, "bf16"),
])
def test_forward_varlen_matches_each_sequence(lengths, H, dk, dv, chunk, dtype):
    from log_linear_attention_gb300 import binding
    seqs, packed, cu, max_T = packed_problem(lengths, H, dk, dv, dtype, seed=len(lengths) + dk)
    q, k, v, la, lam = to_dev(packed, seqs, dtype)
    cu_d = torch.from_numpy(cu).cuda()
    out = binding.forward_varlen(q, k, v, la, lam, cu_d, max_T, chunk)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = out.float().cpu().numpy()
    tol = 1e-4 if dtype == "f32" else 2e-2
    for b, x in enumerate(seqs):
        ref = oracle.explicit(x.q, x.k, x.v, x.log_a, x.lam)[0]
        assert rel_err_per_head(got[:, cu[b]:cu[b + 1]], ref) <= tol, b


@pytest.mark.parametrize("lengths,H,dk", [([128, 1, 383, 2048, 129], 3, 64), ([3000, 130, 64, 255], 2, 128)])
def test_forward_varlen_tensor_core_ragged(lengths, H, dk):
    """bf16 with dv = 64 walks each sequence's own tiles of the packed layout on the tensor-core
    kernels (no padded copy): ragged last tiles, sequences shorter than a tile, dk = 64 and 128."""
    from log_linear_attention_gb300 import binding
    seqs, packed, cu, max_T = packed_problem(lengths, H, dk, 64, "bf16", seed=3 * len(lengths) + dk)
    q, k, v, la, lam = to_dev(packed, seqs, "bf16")
    out = binding.forward_varlen(q, k, v, la, lam, torch.from_numpy(cu).cuda(), max_T, 64)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = out.float().cpu().numpy()
    for b, x in enumerate(seqs):
        fn = oracle.explicit if lengths[b] <= 512 else oracle.recurrent
        ref = fn(x.q, x.k, x.v, x.log_a, x.lam)[0]
        assert rel_err_per_head(got[:, cu[b]:cu[b + 1]], ref) <= 2e-2, b


def test_forward_varlen_empty_sequences():
    """Zero-length sequences in cu_seqlens own no rows and no tiles; the others are unaffected."""
    from log_linear_attention_gb300 import binding
    lengths = [300, 129]
    seqs, packed, cu2, max_T = packed_problem(lengths, 2, 128, 64, "bf16", seed=41)
    q, k, v, la, lam = to_dev(packed, seqs, "bf16")
    cu = np.array([0, 0, 300, 300, 429, 429], dtype=np.int32)
    out = binding.forward_varlen(q, k, v, la, lam, torch.from_numpy(cu).cuda(), max_T, 64)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = out.float().cpu().numpy()
    for b, x in zip((1, 3), seqs):
        ref = oracle.explicit(x.q, x.k, x.v, x.log_a, x.lam)[0]
        assert rel_err_per_head(got[:, cu[b]:cu[b + 1]], ref) <= 2e-2, b


def held_levels(pos, Lmax):
    return [0] + [l for l in range(1, Lmax) if (pos >> (l - 1)) & 1]


@pytest.mark.parametrize("lengths,H,dk,dv,dtype", [
    ([1, 37, 128, 300], 2, 16, 16, "f32"),
    ([100, 640, 0, 257], 2, 128, 64, "bf16"),
])
def test_prefill_state_varlen_then_decode(lengths, H, dk, dv, dtype):
    """States after each sequence match the oracle's recurrence, and decode steps continuing each
    sequence from its own length reproduce the explicit form of the longer sequence."""
    from log_linear_attention_gb300 import binding
    extra = 3
    full = [n + extra for n in lengths]
    seqs_full, _, _, _ = packed_problem(full, H, dk, dv, dtype, seed=7)
    # the prompts are the first `lengths[b]` tokens of each full sequence
    max_T = max(lengths)
    L = inputs.num_levels(max(full))
    Lmax = L + 1

    def prompt(x, n, name):
        return getattr(x, name)[0][:, :n]

    packed_np = {n: np.concatenate([prompt(x, lengths[b], n) for b, x in enumerate(seqs_full)], axis=1)
                 for n in ("q", "k", "v", "log_a")}
    if dtype == "bf16":
        kb = np.concatenate([x.bits["k"][0][:, :lengths[b]] for b, x in enumerate(seqs_full)], axis=1)
        vb = np.concatenate([x.bits["v"][0][:, :lengths[b]] for b, x in enumerate(seqs_full)], axis=1)
        k, v = torch_bf16(kb, "cuda"), torch_bf16(vb, "cuda")
    else:
        k, v = (torch.from_numpy(np.ascontiguousarray(packed_np[n], dtype=np.float32)).cuda() for n in ("k", "v"))
    la = torch.from_numpy(np.ascontiguousarray(packed_np["log_a"], dtype=np.float32)).cuda()
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    n = len(lengths)
    states = torch.full((n, H, Lmax, dk, dv), float("nan"), dtype=torch.float32, device="cuda")
    binding.prefill_state_varlen(k, v, la, torch.from_numpy(cu).cuda(), max_T, states)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got = states.cpu().numpy()
    for b, x in enumerate(seqs_full):
        if lengths[b] == 0:
            assert np.isnan(got[b]).all()
            continue
        ref = np.zeros((1, H, Lmax, dk, dv))
        lam1 = np.ones((1, H, Lmax))
        for t in range(lengths[b]):
            oracle.decode_step(x.q[:, :, t], x.k[:, :, t], x.v[:, :, t], x.log_a[:, :, t], lam1, ref, np.full(1, t))
        for l in held_levels(lengths[b] - 1, Lmax):
            d = np.abs(got[b, :, l] - ref[0, :, l]).max() / max(np.abs(ref[0, :, l]).max(), 1e-30)
            assert d <= 1e-4, (b, l, d)
    # continue every sequence from its own position
    tol = 1e-4 if dtype == "f32" else 2e-2
    for step in range(extra):
        def tok(name, dt):
            rows = [getattr(x, name)[0][:, lengths[b] + step] for b, x in enumerate(seqs_full)]
            return np.stack(rows, axis=0)
        if dtype == "bf16":
            qd, kd, vd = (torch_bf16(np.stack([x.bits[nm][0][:, lengths[b] + step] for b, x in enumerate(seqs_full)], 0),
                                     "cuda") for nm in ("q", "k", "v"))
        else:
            qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(tok(nm, None), dtype=np.float32)).cuda()
                          for nm in ("q", "k", "v"))
        lad = torch.from_numpy(np.ascontiguousarray(tok("log_a", None), dtype=np.float32)).cuda()
        lamd = torch.from_numpy(np.ascontiguousarray(np.stack([x.lam[0][:, lengths[b] + step, :Lmax] if x.lam.shape[3] >= Lmax
                                                               else np.pad(x.lam[0][:, lengths[b] + step], ((0, 0), (0, Lmax - x.lam.shape[3])))
                                                               for b, x in enumerate(seqs_full)], 0), dtype=np.float32)).cuda()
        tpos = torch.tensor([lengths[b] + step for b in range(n)], dtype=torch.int64, device="cuda")
        o = binding.decode_step(qd, kd, vd, lad, lamd, states, tpos).float().cpu().numpy()
        for b, x in enumerate(seqs_full):
            if lengths[b] == 0:
                continue
            ref = oracle.explicit_rows(x.q, x.k, x.v, x.log_a, x.lam, 0, 0, [lengths[b] + step])[0]
            for h in range(H):
                r = oracle.explicit_rows(x.q, x.k, x.v, x.log_a, x.lam, 0, h, [lengths[b] + step])[0]
                assert np.abs(o[b, h] - r).max() / np.abs(r).max() <= tol, (b, h, step)
    assert binding.device_error() == 0


def test_varlen_bad_lengths_are_reported():
    """A sequence longer than max_T is caught on the device: skipped, LLA_ERR_DEVICE reported."""
    from log_linear_attention_gb300 import binding
    H, dk, dv = 1, 16, 16
    total = 96
    q = torch.zeros((H, total, dk), device="cuda")
    la = torch.zeros((H, total), device="cuda")
    lam = torch.ones((H, total, inputs.num_levels(64)), device="cuda")
    cu = torch.tensor([0, 10, 96], dtype=torch.int32, device="cuda")  # second length 86 > max_T 64
    binding.forward_varlen(q, q, q, la, lam, cu, 64, 16)
    assert binding.device_error() == binding.LLA_ERR_DEVICE
    assert binding.device_error() == 0


def test_varlen_bad_lengths_tensor_core_path():
    """The same check on the tensor-core walk (bf16, dk = 128, dv = 64): the over-long sequence is
    skipped (its rows untouched), the error is reported, the valid sequence is correct."""
    from log_linear_attention_gb300 import binding
    seqs, packed, _, max_T = packed_problem([200], 1, 128, 64, "bf16", seed=77)
    q, k, v, la, lam = to_dev(packed, seqs, "bf16")
    # rows 0..199 hold sequence 0; sequence 1 claims rows 200..455, longer than max_T = 200
    pad = lambda x: torch.cat([x, torch.zeros((1, 256) + tuple(x.shape[2:]), dtype=x.dtype, device="cuda")], 1)  # noqa: E731
    q, k, v, la, lam = (pad(x) for x in (q, k, v, la, lam))
    out = torch.full((1, 456, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 200, 456, 456], dtype=torch.int32, device="cuda")
    binding.forward_varlen(q, k, v, la, lam, cu, max_T, 64, out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == binding.LLA_ERR_DEVICE
    assert binding.device_error() == 0
    assert torch.all(out[:, 200:] == 7.0)
    x = seqs[0]
    ref = oracle.explicit(x.q, x.k, x.v, x.log_a, x.lam)[0]
    assert rel_err_per_head(out[:, :200].float().cpu().numpy(), ref) <= 2e-2
