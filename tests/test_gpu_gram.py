"""Kronecker factors from samples on the GPU (bakron_gram, bakron_sq_norms,
bakron_damp) against the oracle ("BaKron: Efficient Quantization with
Kronecker-Factored Hessians", Sec. 4.2, App. A.2, App. D).

Tolerance, from the arithmetic: every bf16 x bf16 product is exact in fp32;
the tensor cores add the products of an entry in fp32 over segments of at
most SEG = 2048 samples, and the kernel adds the nseg = ceil(N / SEG)
segment sums into a running fp32 sum and scales it once by alpha.  So entry
(i, j) is within (2 (min(N, SEG) + 16) + nseg) 2^-24 alpha sum_t
|w_t x_it x_jt| of the exact value (the sequential fp32 summation bound of
one segment, doubled for the order inside the MMA; one rounding per
segment added and one for the scaling); with weights, the bf16 split of
w_t x_t leaves 2^-16 relative per term more.  The typical error is also checked: Frobenius norm within
1e-5 relative, at every N up to the 65536 samples of the full-size case,
plus (with weights) the 2^-16 of alpha |X| diag(|w|) |X|^T the split may
leave."""

import numpy as np
import pytest

import oracle as O
from workloads.activations import make_sample_config, make_samples

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
SEG = 2048  # samples per fp32 accumulation segment of bakron_gram


@pytest.fixture(scope="module")
def bk():
    import torch

    import kronecker_hessian_gptq_gb300 as bk
    from kronecker_hessian_gptq_gb300 import build as b

    b.build()
    bk.load_library()
    torch.cuda.init()
    return bk


def _bf16_dev(bits, ld=None):
    """A bf16 CUDA tensor holding the bit patterns (rows padded to ld)."""
    import torch

    d, N = bits.shape
    ld = (N + 7) // 8 * 8 if ld is None else ld
    buf = np.zeros((d, ld), dtype=np.uint16)
    buf[:, :N] = bits
    t = torch.from_numpy(buf.view(np.int16)).cuda().view(torch.bfloat16)
    return t[:, :N]


def _f32_dev(x):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _bound(Xf, w, alpha, weighted, rounded_weights=False):
    """Entrywise bound; rounded_weights: the weights were themselves rounded
    once to fp32 (relative 2^-24 per term more)."""
    A = np.abs(Xf.astype(np.float64))
    aw = A if w is None else A * np.abs(np.asarray(w, np.float64))[None, :]
    S = alpha * (aw @ A.T)
    N = Xf.shape[1]
    nseg = -(-N // SEG)
    rel = (2 * (min(N, SEG) + 16) + nseg) * U + (2.0 ** -16 if weighted else 0.0) + (U if rounded_weights else 0.0)
    return S * rel + 1e-30


def _split_norm(Xf, w, alpha):
    """Frobenius norm of the error the bf16 split of w_t x_t may leave: 2^-16
    (two roundings of 2^-17 at most) of alpha |X| diag(|w|) |X|^T."""
    A = np.abs(Xf.astype(np.float64))
    return 2.0 ** -16 * alpha * float(np.linalg.norm((A * np.abs(np.asarray(w, np.float64))[None, :]) @ A.T))


def _check(G, ref, bound, frob_extra=0.0):
    """Entrywise bound; Frobenius error within 1e-5 relative (plus, with
    weights, what their bf16 split may leave)."""
    err = np.abs(G.astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / bound).max())
    assert np.linalg.norm(G - ref) <= 1e-5 * np.linalg.norm(ref) + frob_extra + 1e-30
    assert np.array_equal(G, G.T)


@pytest.mark.parametrize("d,N", [(1, 1), (5, 7), (64, 64), (128, 100), (130, 1000), (257, 333), (64, 2100), (130, 5000)])
@pytest.mark.parametrize("weighted", [False, True])
def test_gram_against_oracle(bk, d, N, weighted):
    import torch

    s = make_samples(d, 3, N, seed=d * 7 + N)
    Xf = s.a_f32
    w = O.squared_norms(s.b_f32).astype(np.float32) if weighted else None
    ld = (N + 7) // 8 * 8 + (8 if d % 2 else 0)  # padded rows, sometimes wider than needed
    G, st = bk.gram(_bf16_dev(s.a_bits, ld), None if w is None else _f32_dev(w))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.weighted_gram(Xf, w)
    extra = _split_norm(Xf, w, 1.0 / N) if weighted else 0.0
    _check(G.cpu().numpy(), ref, _bound(Xf, w, 1.0 / N, weighted), extra)


def test_gram_accumulates_batches(bk):
    """Two batches with beta = 1 and alpha = 1 / (total samples): the mean
    over all samples."""
    import torch

    s = make_samples(150, 2, 700, seed=3)
    G, _ = bk.gram(_bf16_dev(s.a_bits[:, :300]), alpha=1.0 / 700)
    G, st = bk.gram(_bf16_dev(s.a_bits[:, 300:]), alpha=1.0 / 700, beta=1.0, out=G)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.weighted_gram(s.a_f32)
    _check(G.cpu().numpy(), ref, _bound(s.a_f32, None, 1.0 / 700, False))


def test_shampoo_one_step_end_to_end(bk):
    """Shampoo factors from the GPU's squared norms and weighted Grams against
    the oracle's power iteration (one step from the identity)."""
    import torch

    s = make_samples(96, 80, 500, seed=11)
    a, b = _bf16_dev(s.a_bits), _bf16_dev(s.b_bits)
    wa, wb = bk.sq_norms(b), bk.sq_norms(a)  # weights of a a^T: |b|^2; of b b^T: |a|^2
    A, _ = bk.gram(a, wa)
    B, _ = bk.gram(b, wb)
    torch.cuda.synchronize()
    assert np.allclose(wa.cpu().numpy(), O.squared_norms(s.b_f32), rtol=1e-6, atol=0)
    Ao, Bo = O.shampoo_factors(s.a_f32, s.b_f32, 1)
    # the GPU's weights are the squared norms rounded once to fp32
    wa_, wb_ = O.squared_norms(s.b_f32), O.squared_norms(s.a_f32)
    _check(A.cpu().numpy(), Ao, _bound(s.a_f32, wa_, 1 / 500, True, rounded_weights=True), _split_norm(s.a_f32, wa_, 1 / 500))
    _check(B.cpu().numpy(), Bo, _bound(s.b_f32, wb_, 1 / 500, True, rounded_weights=True), _split_norm(s.b_f32, wb_, 1 / 500))


def test_damp_against_oracle(bk):
    import torch

    rng = np.random.default_rng(2)
    X = rng.standard_normal((300, 400))
    G = (X @ X.T / 400).astype(np.float32)
    Gd = bk.damp(_f32_dev(G), 0.5)
    torch.cuda.synchronize()
    ref = O.damp(G.astype(np.float64), 0.5)
    assert np.allclose(Gd.cpu().numpy(), ref, rtol=2e-7, atol=1e-6)
    off = ~np.eye(300, dtype=bool)
    assert np.array_equal(Gd.cpu().numpy()[off], G[off])


def test_gram_full_size_sampled_entries(bk):
    """The 4096-feature input side with 65536 samples (K-FAC), every diagonal
    entry and 4096 sampled entries against the oracle's exact dot products."""
    import torch

    s = make_sample_config("g3")
    G, st = bk.gram(_bf16_dev(s.a_bits))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    G = G.cpu().numpy()
    Xf = s.a_f32.astype(np.float64)
    rng = np.random.default_rng(0)
    ii = np.concatenate([np.arange(s.n), rng.integers(0, s.n, 4096)])
    jj = np.concatenate([np.arange(s.n), rng.integers(0, s.n, 4096)])
    ref = np.einsum("kt,kt->k", Xf[ii], Xf[jj]) / s.N
    nseg = -(-s.N // SEG)
    bnd = np.einsum("kt,kt->k", np.abs(Xf[ii]), np.abs(Xf[jj])) / s.N * (2 * (min(s.N, SEG) + 16) + nseg) * U
    err = np.abs(G[ii, jj] - ref)
    rel = np.linalg.norm(err) / np.linalg.norm(ref)
    worst = float((err / bnd).max())
    assert np.all(err <= bnd), (worst, rel)
    # fp32 accumulation over 2048-sample segments, then 32 segment sums (measured 5.2e-6)
    print(f"\ngram 4096 x 65536: Frobenius error {rel:.3g} relative, worst entry at {worst:.3g} of its bound")
    assert rel <= 1e-5, (worst, rel)
    assert np.array_equal(G, G.T)
