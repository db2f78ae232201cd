"""Kronecker factors of a Hessian from samples (oracle; test infrastructure
only).

"BaKron: Efficient Quantization with Kronecker-Factored Hessians", Sec. 4.2
and App. A.2: a Hessian of the form H = E[a a^T (x) b b^T] (a the input of a
linear unit, b the backpropagated output side) is approximated by a
Kronecker product A (x) B in one of two ways:

* K-FAC style: A = E[a a^T], B = E[b b^T] (the expectation pulled apart);
* Shampoo style: the best Frobenius approximation, whose factors are the top
  singular pair of the rearranged matrix R(H) = E[vec(a a^T) vec(b b^T)^T]
  (Van Loan and Pitsianis), found by power iteration
      A^(i+1) = E[(b^T B^(i) b) a a^T],   B^(i+1) = E[(a^T A^(i) a) b b^T],
  one step from A^(0) = I, B^(0) = I giving E[|b|^2 a a^T], E[|a|^2 b b^T].

App. D regularizes every Gram matrix by adding 0.5 times its mean diagonal
value to the diagonal.

Conventions (the reading used): the samples are the columns of a (n x N) and
b (m x N); an expectation is the plain mean over the N samples (the solver is
invariant under scaling the factors, so the normalization only fixes the
numbers); all arithmetic in float64.
"""

from __future__ import annotations

import numpy as np


def weighted_gram(X, w=None) -> np.ndarray:
    """(1/N) sum_t w_t x_t x_t^T for the columns x_t of X (d x N); w None: all ones."""
    X = np.asarray(X, dtype=np.float64)
    N = X.shape[1]
    if N == 0:
        raise ValueError("at least one sample")
    Xw = X if w is None else X * np.asarray(w, dtype=np.float64)[None, :]
    return (Xw @ X.T) / N


def kfac_factors(a, b):
    """K-FAC-style factors (E[a a^T], E[b b^T])."""
    return weighted_gram(a), weighted_gram(b)


def shampoo_factors(a, b, iterations: int = 1):
    """Shampoo-style factors after `iterations` power-iteration steps from
    (I, I), both factors updated from the previous iterate."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    A = np.eye(a.shape[0])
    B = np.eye(b.shape[0])
    for _ in range(iterations):
        wa = np.einsum("it,ij,jt->t", b, B, b)  # b_t^T B b_t, the weight of a_t a_t^T
        wb = np.einsum("it,ij,jt->t", a, A, a)  # a_t^T A a_t
        A, B = weighted_gram(a, wa), weighted_gram(b, wb)
    return A, B


def damp(G, rel: float = 0.5) -> np.ndarray:
    """G + rel * mean(diag(G)) * I (App. D uses rel = 0.5)."""
    G = np.asarray(G, dtype=np.float64)
    return G + rel * np.mean(np.diag(G)) * np.eye(G.shape[0])


def squared_norms(Y) -> np.ndarray:
    """|y_t|^2 of the columns of Y: the one-step Shampoo weights."""
    Y = np.asarray(Y, dtype=np.float64)
    return np.einsum("it,it->t", Y, Y)
