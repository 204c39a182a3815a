"""Pins of the MXFP8 reading's quantisation AXES (CPU).

MXFP8 keeps one power-of-two scale per 32 contiguous elements along a GEMM's reduction
dimension (the MXFP8 workload of the layer; page "Mixture-of-Kittens; MoE megakernel", key
points: BF16 and MXFP8).  On ordinary data the block a value falls in barely matters: E4M3 is a
floating-point format, so a block's scale only changes a value's rounding once that value sits
more than about 2^15 below its block's largest one (it drops into the subnormal codes).  These
pins therefore plant an outlier 2^18 times the rest and check WHICH values it coarsens, through
the oracle's public functions: an outlier coarsens exactly the other values of its own block
along the reduction dimension of the GEMM that reads the tensor, and nothing along the other
axis.  Quantising any operand along the wrong axis (or not at all) fails one of them.

Fixture: 32 tokens, each a one-hot row of x in its own 32-block of d (token t at column 32 t,
with a value a_t in [0.7, 1.6)), so g[t] and u[t] read rows 32 t of W_gate and W_up only; two
more 32-blocks of d (columns 1024..1087) hold no token.  One expert, k = 1, no shared expert.
"""

import numpy as np

import oracle
from oracle.moe import _mx_weight

T, D, F = 32, 1088, 64
BIG = 2.0 ** 18
T0 = 5                 # the token that carries the planted value
I0, I1 = 1024 + 5, 1024 + 9   # two columns of d in a block no token uses
F0, F1 = 7, 9          # two columns of F in the same 32-block
J0, J1 = 100, 105      # two columns of d in the same 32-block


def _fixture(seed):
    rng = np.random.default_rng(seed)
    x = np.zeros((T, D))
    x[np.arange(T), 32 * np.arange(T)] = rng.uniform(0.7, 1.6, size=T)
    Wg = rng.standard_normal((D, F)) * 0.5
    Wu = rng.standard_normal((D, F)) * 0.5
    Wd = rng.standard_normal((F, D)) * 0.2
    dY = rng.standard_normal((T, D))
    return x, Wg, Wu, Wd, dY


IDX = np.zeros((T, 1), dtype=np.int32)   # every token on expert 0, k = 1
W1 = np.ones((T, 1))


def _fwd(x, Wg, Wu, Wd):
    return oracle.moe_forward_mxfp8(x, Wg[None], Wu[None], Wd[None], None, IDX, W1)


def _bwd(x, dY, Wg, Wu, Wd):
    Wr = np.zeros((D, 1))
    return oracle.moe_backward_mxfp8(x, dY, Wr, Wg[None], Wu[None], Wd[None], None,
                                     np.zeros((T, 1)), IDX)


def _same(a, b):
    return np.allclose(a, b, rtol=1e-12, atol=1e-12 * max(np.abs(b).max(), 1e-300))


def _moved(a, b):
    return np.abs(a - b).max() > 1e-6 * np.abs(b).max()


def test_weight_quantiser_blocks_run_along_the_reduction_dimension():
    """_mx_weight(W[K, N]): an outlier at (k0, n0) coarsens its 31 neighbours of column n0 in the
    same 32-row block of K, and no value of row k0 (the N direction)."""
    rng = np.random.default_rng(0)
    W = rng.standard_normal((64, 96))
    k0, n0 = 37, 50
    W1 = W.copy()
    W1[k0, n0] = BIG * np.abs(W).max()
    q0, q1 = _mx_weight(W), _mx_weight(W1)
    blk = [k for k in range(32, 64) if k != k0]
    assert (q1[blk, n0] != q0[blk, n0]).sum() >= 28           # coarsened along K
    assert (q1[k0, np.arange(96) != n0] == q0[k0, np.arange(96) != n0]).all()   # not along N
    assert (q1[:32] == q0[:32]).all() and (q1[:, np.arange(96) != n0] == q0[:, np.arange(96) != n0]).all()


# ---------------------------------------------------------------- forward quantisation points

def test_forward_gate_weight_along_d():
    """An outlier at W_gate[i0, f0] with x[:, i0] = 0 still changes token t0's output: it coarsens
    W_gate[32 t0, f0], in the same 32-block of d (the gate GEMM's reduction dimension).  Along F
    it would only touch row i0, which no token reads."""
    x, Wg, Wu, Wd, _ = _fixture(1)
    i0 = 32 * T0 + 3
    Wg1 = Wg.copy()
    Wg1[i0, F0] = BIG * np.abs(Wg).max()
    y0, y1 = _fwd(x, Wg, Wu, Wd), _fwd(x, Wg1, Wu, Wd)
    assert _moved(y1[T0], y0[T0])
    others = np.arange(T) != T0
    assert _same(y1[others], y0[others])


def test_forward_up_weight_along_d():
    x, Wg, Wu, Wd, _ = _fixture(2)
    i0 = 32 * T0 + 3
    Wu1 = Wu.copy()
    Wu1[i0, F0] = BIG * np.abs(Wu).max()
    y0, y1 = _fwd(x, Wg, Wu, Wd), _fwd(x, Wg, Wu1, Wd)
    assert _moved(y1[T0], y0[T0])
    others = np.arange(T) != T0
    assert _same(y1[others], y0[others])


def test_forward_down_weight_along_F():
    """h[:, f0] = 0 (W_up column f0 zero); an outlier at W_down[f0, j0] changes output column j0
    only, by coarsening W_down[f, j0] for the other f of its 32-block of F (the down GEMM's
    reduction dimension).  Along d it would only touch row f0, which h never weights."""
    x, Wg, Wu, Wd, _ = _fixture(3)
    Wu[:, F0] = 0.0
    Wd1 = Wd.copy()
    Wd1[F0, J0] = BIG * np.abs(Wd).max()
    y0, y1 = _fwd(x, Wg, Wu, Wd), _fwd(x, Wg, Wu, Wd1)
    assert _moved(y1[:, J0], y0[:, J0])
    others = np.arange(D) != J0
    assert _same(y1[:, others], y0[:, others])


def test_forward_x_along_d():
    """A large x[t0, i0] in token t0's own 32-block of d (rows i0 of both weights zero, so it adds
    nothing itself) coarsens x[t0, 32 t0] and so changes token t0's output, and only that.  Along
    tokens its block would hold no other nonzero value."""
    x, Wg, Wu, Wd, _ = _fixture(4)
    i0 = 32 * T0 + 1
    Wg[i0, :] = Wu[i0, :] = 0.0
    x1 = x.copy()
    x1[T0, i0] = BIG * 2.0
    y0, y1 = _fwd(x, Wg, Wu, Wd), _fwd(x1, Wg, Wu, Wd)
    assert _moved(y1[T0], y0[T0])
    others = np.arange(T) != T0
    assert _same(y1[others], y0[others])


def test_forward_h_along_F():
    """A large h[t0, f0] (W_up[32 t0, f0] scaled up) coarsens token t0's other h values in its
    32-block of F and no other token's h: every other token's output is unchanged.  Along tokens
    it would coarsen h[t, f0] of every token of its block."""
    x, Wg, Wu, Wd, _ = _fixture(5)
    Wg[32 * T0, F0] = 2.0
    Wu1 = Wu.copy()
    Wu1[32 * T0, F0] = BIG * np.abs(Wu).max()
    y0, y1 = _fwd(x, Wg, Wu, Wd), _fwd(x, Wg, Wu1, Wd)
    assert _moved(y1[T0], y0[T0])
    others = np.arange(T) != T0
    assert _same(y1[others], y0[others])


# ---------------------------------------------------------------- backward quantisation points

def test_backward_down_weight_along_d():
    """u (hence h) of every token is one-hot at f1.  An outlier at W_down[f0, j0], f0 in f1's
    32-block of F, leaves every router-weight gradient dw = <a, h> = a[:, f1] h[:, f1] unchanged:
    a = dY W_down^T quantises W_down along d (row f0 only).  Along F it would coarsen
    W_down[f1, j0]."""
    x, Wg, Wu, Wd, dY = _fixture(6)
    Wu[:, :] = 0.0
    Wu[32 * np.arange(T), F1] = 1.0
    Wd1 = Wd.copy()
    Wd1[F0, J0] = BIG * np.abs(Wd).max()
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x, dY, Wg, Wu, Wd1)
    assert np.abs(r0["dw"]).min() > 0
    assert _same(r1["dw"], r0["dw"])


def test_backward_gate_and_up_weights_along_F():
    """dX = q(dG) q(W_gate)^T + q(dU) q(W_up)^T reduces over F: an outlier at W_gate[i0, f0] (or
    W_up[i0, f0]) in a block of d that no token reads changes dX[:, i0] and leaves dX[:, i1]
    unchanged.  Along d it would coarsen W_gate[i1, f0]."""
    x, Wg, Wu, Wd, dY = _fixture(7)
    r0 = _bwd(x, dY, Wg, Wu, Wd)
    for which in ("gate", "up"):
        Wg1, Wu1 = Wg.copy(), Wu.copy()
        W = Wg1 if which == "gate" else Wu1
        W[I0, F0] = BIG * np.abs(W).max()
        r1 = _bwd(x, dY, Wg1, Wu1, Wd)
        assert _moved(r1["dX"][:, I0], r0["dX"][:, I0]), which
        assert _same(r1["dX"][:, I1], r0["dX"][:, I1]), which


def test_backward_dY_along_tokens_for_the_down_weight_gradient():
    """dW_down = q_t(w h)^T q_t(dY) reduces over tokens: a large dY[t0, j0] changes dW_down[:, j0]
    and leaves dW_down[:, j1] (same 32-block of d) unchanged.  Along d it would coarsen
    dY[t0, j1]."""
    x, Wg, Wu, Wd, dY = _fixture(8)
    dY1 = dY.copy()
    dY1[T0, J0] = BIG * np.abs(dY).max()
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x, dY1, Wg, Wu, Wd)
    assert _moved(r1["dW_down"][0][:, J0], r0["dW_down"][0][:, J0])
    assert _same(r1["dW_down"][0][:, J1], r0["dW_down"][0][:, J1])


def test_backward_x_along_tokens_for_the_gate_and_up_weight_gradients():
    """dW_gate = q_t(x)^T q_t(dG) reduces over tokens: with weight rows i0, i1 zero (the forward
    ignores those columns of x), a large x[t0, i0] leaves dW_gate[i1] and dW_up[i1] unchanged
    (column i1 of x has one nonzero token).  Along d it would coarsen x[t0, i1]."""
    x, Wg, Wu, Wd, dY = _fixture(9)
    Wg[1024:, :] = Wu[1024:, :] = 0.0
    x[T0, I1] = 0.37
    x1 = x.copy()
    x1[T0, I0] = BIG
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x1, dY, Wg, Wu, Wd)
    assert np.abs(r0["dW_gate"][0][I1]).max() > 0
    assert _moved(r1["dW_gate"][0][I0], r0["dW_gate"][0][I0])
    assert _same(r1["dW_gate"][0][I1], r0["dW_gate"][0][I1])
    assert _same(r1["dW_up"][0][I1], r0["dW_up"][0][I1])


def test_backward_dG_and_dU_along_tokens():
    """W_down row f0 scaled by 2^18 scales a[:, f0], hence dG[:, f0] and dU[:, f0], uniformly along
    tokens: the weight gradients of the other columns f1 of its block of F are unchanged.  Along F
    the large dG[t, f0] would coarsen dG[t, f1] of every token."""
    x, Wg, Wu, Wd, dY = _fixture(10)
    Wd1 = Wd.copy()
    Wd1[F0, :] *= BIG
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x, dY, Wg, Wu, Wd1)
    for key in ("dW_gate", "dW_up"):
        assert _moved(r1[key][0][:, F0], r0[key][0][:, F0]), key
        assert _same(r1[key][0][:, F1], r0[key][0][:, F1]), key


def test_backward_wh_along_tokens():
    """A large h[t0, f0] (W_up[32 t0, f0] scaled up) changes dW_down[f0] only: w h is quantised
    along tokens for dW_down = q_t(w h)^T q_t(dY), so h[t0, f1] keeps its value.  Along F it would
    coarsen h[t0, f1] and change dW_down[f1]."""
    x, Wg, Wu, Wd, dY = _fixture(11)
    Wg[32 * T0, F0] = 2.0
    Wu1 = Wu.copy()
    Wu1[32 * T0, F0] = BIG * np.abs(Wu).max()
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x, dY, Wg, Wu1, Wd)
    assert _moved(r1["dW_down"][0][F0], r0["dW_down"][0][F0])
    assert _same(r1["dW_down"][0][F1], r0["dW_down"][0][F1])


def test_backward_dY_along_d_and_dG_dU_along_F():
    """A large dY[t0, j0] changes only token t0's per-token gradients: a = q_d(dY) q_d(W_down)^T
    quantises dY along d (row t0), and dX = q_F(dG) q_F(W_gate)^T + q_F(dU) q_F(W_up)^T quantises
    dG and dU along F (row t0's large values stay in row t0).  Every other token's dX and dw is
    unchanged; along tokens either would coarsen the other tokens of t0's block."""
    x, Wg, Wu, Wd, dY = _fixture(12)
    dY1 = dY.copy()
    dY1[T0, J0] = BIG * np.abs(dY).max()
    r0, r1 = _bwd(x, dY, Wg, Wu, Wd), _bwd(x, dY1, Wg, Wu, Wd)
    others = np.arange(T) != T0
    assert _moved(r1["dX"][T0], r0["dX"][T0])
    assert _same(r1["dX"][others], r0["dX"][others])
    assert _same(r1["dw"][others], r0["dw"][others])


def test_backward_forward_values_use_the_forward_axes():
    """The backward differentiates the MXFP8 forward's g and u, whose weights are quantised along
    d: an outlier at W_gate[i0, f0] (or W_up) with x[:, i0] = 0 moves token t0's router-weight
    gradient dw = <a, h> through the coarsened W[32 t0, f0].  Along F it would touch row i0 only,
    which no token reads in the forward."""
    x, Wg, Wu, Wd, dY = _fixture(13)
    i0 = 32 * T0 + 3
    r0 = _bwd(x, dY, Wg, Wu, Wd)
    for which in ("gate", "up"):
        Wg1, Wu1 = Wg.copy(), Wu.copy()
        W = Wg1 if which == "gate" else Wu1
        W[i0, F0] = BIG * np.abs(W).max()
        r1 = _bwd(x, dY, Wg1, Wu1, Wd)
        others = np.arange(T) != T0
        assert _moved(r1["dw"][T0], r0["dw"][T0]), which
        assert _same(r1["dw"][others], r0["dw"][others]), which
