"""Plain fp64 CPU oracle for fused linear cross-entropy and the standalone row-wise CE kernel.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this module: only the
tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no code with the CUDA
library and imports nothing from the package.

Every function here is the textbook definition written out in float64, in the notation of
"Fused Linear Cross-Entropy: The Math, the Memory Wall, and Two Ways Around It" (p1) and
"Greyhound -- Cross-Entropy" (p3).  Inputs are bf16 bit patterns (uint16) or float arrays; they are
widened exactly to float64 before any arithmetic.

Definitions followed (page, section):
  * logits z = W . hidden[t] (+ b), p = softmax(z), l_t = -z_y + LSE(z)       p1 "The setting"
  * L = (1/n_valid) sum_t l_t [y_t != -100] (mean); the plain sum for "sum"   p1 "The setting";
                                                                              p2 "Forward pass" (mean, sum)
  * dl_t/dz = softmax(z) - onehot(y_t)  (boxed identity)                      p1 "The identity that makes
                                                                                 fused fwbw possible"
  * LSE = max z + log sum exp(z - max z)                                      same section, consequence 3
  * dlogits[t,:] = (1/n_valid) [y_t != -100] (softmax(z_t) - onehot(y_t));
    grad_input = dlogits . W;  grad_W = dlogits^T . hidden;
    grad_b = sum_t dlogits[t,:]                                               p1 "From dlogits to
                                                                                 grad_input and grad_W"
  * z_i = LSE_i^2 (z-loss), its gradient scales the softmax term before the
    target column is adjusted                                                 p3 formulas, "Loss and
                                                                                 gradient together"
  * loss = ce_sum / max(n_valid, 1)                                           p3 "Usage" (raw helper)

Readings where the pages are silent:
  * with z-loss in the fused loss, l_t = LSE_t - z_y + z_loss * LSE_t^2, so the gradient row is
    p * (1 + 2 z_loss LSE_t) - onehot(y_t);
  * n_valid = 0 gives loss 0 and all-zero gradients (the clamp of p3 "Usage");
  * the per-row entropy that verl's forward kernel returns (p1 "Strategy 2", entropy_b) is read as the
    Shannon entropy of softmax(z_t), computed for every row whatever its target;
  * reduction "none" returns the per-token losses; its gradients are those of sum_t g_t l_t for an
    upstream gradient g (PyTorch's convention for an unreduced loss), and every gradient is
    multiplied by the scalar upstream gradient of the reduced loss (the d_out / grad_scale factor of
    p2 "Breakdown: Backward Pass", step 4);
  * a target outside [0, V) that is not ignore_index is treated as ignored;
  * z_sum of the standalone CE is the unscaled sum of LSE^2 over valid rows.
  * logit_avg (p2 "Forward pass", the by-product of the LSE kernel that keys the vocabulary sort) is the
    mean of z[t, n] over all BT rows of the batch, ignored rows included (the forward kernel sees every
    row); an empty batch gives 0 (+ b);
  * the vocabulary order of p2 "Vocabulary Sorting" is by average logit, largest first, equal keys in
    increasing vocabulary index (a stable sort).

Rows are processed in blocks only to bound memory: the loss is a sum over tokens and both gradients
are sums of per-token terms, and p1 ("The identity ...", consequence 2) states that this sum commutes
with chunking over tokens.  No other blocking, fusion or reordering is done.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "widen", "logits", "lse", "flce_reference", "flce_dlogits", "flce_lse", "flce_sampled", "flce_reference_loops",
    "ce_reference", "ce_reference_loops", "logit_avg", "vocab_order",
]


def widen(x) -> np.ndarray:
    """bf16 bit patterns (uint16) or any float array -> float64, exactly (a float64 array is used as is)."""
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def logits(hidden, W, bias=None) -> np.ndarray:
    """z = hidden . W^T (+ b) in float64 (p1 "The setting": z = W . hidden[t])."""
    z = widen(hidden) @ widen(W).T
    if bias is not None:
        z = z + widen(bias)[None, :]
    return z


def lse(z: np.ndarray) -> np.ndarray:
    """Row-wise log-sum-exp, LSE = max z + log sum exp(z - max z) (p1, consequence 3)."""
    m = np.max(z, axis=-1)
    return m + np.log(np.sum(np.exp(z - m[..., None]), axis=-1))


def _valid_mask(target: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    t = np.asarray(target, dtype=np.int64)
    return (t != ignore_index) & (t >= 0) & (t < V)


def _scale(n_valid: int, reduction: str) -> float:
    if reduction == "mean":
        return 1.0 / max(n_valid, 1)
    if reduction in ("sum", "none"):
        return 1.0
    raise ValueError(f"reduction must be 'mean', 'sum' or 'none', got {reduction!r}")


def flce_reference(hidden, W, target, bias=None, ignore_index: int = -100, reduction: str = "mean",
                   z_loss: float = 0.0, want_grads: bool = True, row_block: int = 512, grad_scale: float = 1.0,
                   grad_loss_per_token=None) -> dict:
    """Loss and gradients of fused linear cross-entropy, straight from the definitions.

    Returns a dict with ``loss`` (float), ``n_valid`` (int), ``lse`` [BT], ``loss_per_token`` [BT]
    (l_t on valid rows, 0 elsewhere), ``entropy`` [BT] (the entropy of softmax(z_t) for every row,
    -sum_n p log p = LSE_t - sum_n p_n z_n), and when ``want_grads`` ``grad_input`` [BT, H], ``grad_W`` [V, H],
    ``grad_bias`` [V] (None without a bias), all float64.

    reduction "mean" / "sum": ``loss`` is the reduced loss.  reduction "none": ``loss`` is the plain
    sum of ``loss_per_token`` and the gradients are those of sum_t g_t l_t, with g_t the upstream
    gradient of token t's loss (``grad_loss_per_token``; all ones when None).  Every gradient is
    multiplied by ``grad_scale`` (the upstream gradient of the reduced loss).
    """
    h = widen(hidden)
    w = widen(W)
    b = None if bias is None else widen(bias)
    t = np.asarray(target, dtype=np.int64)
    BT, H = h.shape
    V = w.shape[0]
    valid = _valid_mask(t, V, ignore_index)
    n_valid = int(valid.sum())
    s = _scale(n_valid, reduction)

    loss_terms = []
    lse_all = np.empty(BT)
    ent_all = np.empty(BT)
    u = np.ones(BT) if grad_loss_per_token is None else np.asarray(grad_loss_per_token, dtype=np.float64)
    if want_grads:
        grad_input = np.zeros((BT, H))
        grad_W = np.zeros((V, H))
        grad_b = np.zeros(V) if b is not None else None
    for r0 in range(0, BT, row_block):
        r1 = min(BT, r0 + row_block)
        rows = np.arange(r1 - r0)
        z = h[r0:r1] @ w.T
        if b is not None:
            z += b[None, :]
        m = z.max(axis=1)
        e = np.exp(z - m[:, None])
        denom = e.sum(axis=1)
        L = m + np.log(denom)
        lse_all[r0:r1] = L
        ent_all[r0:r1] = L - (e * z).sum(axis=1) / denom
        v = valid[r0:r1]
        y = np.where(v, t[r0:r1], 0)
        z_y = z[rows, y]
        loss_terms.append(np.where(v, (L - z_y) + z_loss * L * L, 0.0))
        if want_grads:
            p = e / denom[:, None]
            d = p * (1.0 + 2.0 * z_loss * L)[:, None]
            d[rows, y] -= 1.0
            d *= (s * v)[:, None]
            d *= (grad_scale * u[r0:r1])[:, None]
            grad_input[r0:r1] = d @ w
            grad_W += d.T @ h[r0:r1]
            if grad_b is not None:
                grad_b += d.sum(axis=0)
    per_token = np.concatenate(loss_terms) if loss_terms else np.zeros(0)
    loss = s * math.fsum(per_token.tolist()) if loss_terms else 0.0
    out = dict(loss=loss, n_valid=n_valid, lse=lse_all, loss_per_token=per_token, entropy=ent_all)
    if want_grads:
        out.update(grad_input=grad_input, grad_W=grad_W, grad_bias=grad_b)
    return out


def flce_dlogits(hidden, W, target, bias=None, ignore_index: int = -100, reduction: str = "mean",
                 z_loss: float = 0.0) -> np.ndarray:
    """The full [BT, V] dlogits matrix of the fused loss (small cases only): s [y_t valid]
    (softmax(z_t) (1 + 2 z_loss LSE_t) - onehot(y_t)), p1 "From dlogits to grad_input and grad_W"."""
    z = logits(hidden, W, bias)
    t = np.asarray(target, dtype=np.int64)
    V = z.shape[1]
    valid = _valid_mask(t, V, ignore_index)
    s = _scale(int(valid.sum()), reduction)
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    tot = e.sum(axis=1)
    lse_rows = m + np.log(tot)
    d = e / tot[:, None] * (1.0 + 2.0 * z_loss * lse_rows)[:, None]
    rows = np.nonzero(valid)[0]
    d[rows, t[rows]] -= 1.0
    return d * (s * valid)[:, None]


def flce_lse(hidden, W, bias=None, row_block: int = 512) -> np.ndarray:
    """LSE of every row of z = hidden . W^T (+ b), float64, without gradients."""
    h = widen(hidden)
    w = widen(W)
    b = None if bias is None else widen(bias)
    out = np.empty(h.shape[0])
    for r0 in range(0, h.shape[0], row_block):
        z = h[r0:r0 + row_block] @ w.T
        if b is not None:
            z += b[None, :]
        out[r0:r0 + row_block] = lse(z)
    return out


def flce_sampled(hidden, W, target, lse_all, rows, vocab_rows, bias=None, ignore_index: int = -100,
                 reduction: str = "mean", z_loss: float = 0.0) -> dict:
    """Selected outputs of the fused path, given the float64 LSE of every row (from ``flce_lse``).

    * ``loss`` over all rows (needs only LSE and z_y),
    * ``grad_input[rows]``: dlogits rows times W,
    * ``grad_W[vocab_rows]`` and ``grad_bias[vocab_rows]``: the dlogits columns of those vocabulary
      entries (over every token) times hidden.
    All from the same definitions as ``flce_reference``.  The ``*_softmax`` entries are the same rows with
    the onehot term of dlogits left out (only s [y_t valid] softmax(z_t) (1 + 2 z_loss LSE_t)), so that a
    test can tell the softmax part of a gradient row from its target part.
    """
    h = widen(hidden)
    w = widen(W)
    b = None if bias is None else widen(bias)
    t = np.asarray(target, dtype=np.int64)
    BT, H = h.shape
    V = w.shape[0]
    L = np.asarray(lse_all, dtype=np.float64)
    valid = _valid_mask(t, V, ignore_index)
    n_valid = int(valid.sum())
    s = _scale(n_valid, reduction)
    y = np.where(valid, t, 0)

    # z_y for every row: hidden[t] . W[y_t] (+ b[y_t])
    z_y = np.einsum("ij,ij->i", h, w[y])
    if b is not None:
        z_y += b[y]
    loss = s * math.fsum(np.where(valid, (L - z_y) + z_loss * L * L, 0.0).tolist())

    rows = np.asarray(rows, dtype=np.int64)
    z = h[rows] @ w.T
    if b is not None:
        z += b[None, :]
    d = np.exp(z - L[rows][:, None]) * (1.0 + 2.0 * z_loss * L[rows])[:, None]
    gi_soft = (d * (s * valid[rows])[:, None]) @ w
    d[np.arange(len(rows)), y[rows]] -= 1.0
    d *= (s * valid[rows])[:, None]
    gi = d @ w

    vr = np.asarray(vocab_rows, dtype=np.int64)
    zc = h @ w[vr].T                       # [BT, len(vr)] logits columns of the chosen entries
    if b is not None:
        zc += b[vr][None, :]
    dc = np.exp(zc - L[:, None]) * (1.0 + 2.0 * z_loss * L)[:, None]
    dc_soft = dc * (s * valid)[:, None]
    dc -= ((y[:, None] == vr[None, :]) & valid[:, None]).astype(np.float64)
    dc *= (s * valid)[:, None]
    gw = dc.T @ h
    gb = dc.sum(axis=0) if b is not None else None
    return dict(loss=loss, n_valid=n_valid, grad_input_rows=gi, grad_W_rows=gw, grad_bias_rows=gb,
                grad_input_rows_softmax=gi_soft, grad_W_rows_softmax=dc_soft.T @ h,
                grad_bias_rows_softmax=dc_soft.sum(axis=0) if b is not None else None)


def flce_reference_loops(hidden, W, target, bias=None, ignore_index: int = -100,
                         reduction: str = "mean", z_loss: float = 0.0) -> dict:
    """The same definitions with explicit Python loops and ``math`` scalars (tiny shapes only).

    Materialises the full logits, softmax and dlogits matrices element by element, as the naive path
    of p1 "The engineering wall" does, so it can check the vectorised oracle by brute force.
    """
    h = widen(hidden)
    w = widen(W)
    b = None if bias is None else widen(bias)
    t = [int(x) for x in np.asarray(target)]
    BT, H = h.shape
    V = w.shape[0]
    valid = [(y != ignore_index) and (0 <= y < V) for y in t]
    n_valid = sum(valid)
    s = _scale(n_valid, reduction)
    Z = [[math.fsum(float(h[i, k]) * float(w[j, k]) for k in range(H)) + (float(b[j]) if b is not None else 0.0)
          for j in range(V)] for i in range(BT)]
    loss_terms = []
    D = [[0.0] * V for _ in range(BT)]
    lse_rows = []
    for i in range(BT):
        m = max(Z[i])
        L = m + math.log(math.fsum(math.exp(zj - m) for zj in Z[i]))
        lse_rows.append(L)
        if not valid[i]:
            continue
        loss_terms.append(L - Z[i][t[i]] + z_loss * L * L)
        for j in range(V):
            pj = math.exp(Z[i][j] - L)
            D[i][j] = s * (pj * (1.0 + 2.0 * z_loss * L) - (1.0 if j == t[i] else 0.0))
    gi = np.array([[math.fsum(D[i][j] * float(w[j, k]) for j in range(V)) for k in range(H)] for i in range(BT)])
    gw = np.array([[math.fsum(D[i][j] * float(h[i, k]) for i in range(BT)) for k in range(H)] for j in range(V)])
    gb = np.array([math.fsum(D[i][j] for i in range(BT)) for j in range(V)]) if b is not None else None
    return dict(loss=s * math.fsum(loss_terms), n_valid=n_valid, lse=np.array(lse_rows), grad_input=gi,
                grad_W=gw, grad_bias=gb, dlogits=np.array(D))


def ce_reference(logits_, labels, ignore_index: int = -100, z_loss: float = 0.0,
                 row_block: int = 256) -> dict:
    """Standalone row-wise cross-entropy with its logits gradient (p3 "Cross-Entropy").

    Per row: loss_i = LSE(logits_i) - logits_{i, y_i}; z_i = LSE_i^2.  Returns ``ce_sum`` and
    ``z_sum`` over valid rows, ``n_valid``, ``lse`` and ``dlogits`` = p * (1 + 2 z_loss LSE) - onehot(y)
    on valid rows and 0 on ignored rows (the gradient of ce_sum + z_loss * z_sum).
    """
    x = np.asarray(logits_)
    lab = np.asarray(labels, dtype=np.int64)
    B, V = x.shape
    valid = _valid_mask(lab, V, ignore_index)
    y = np.where(valid, lab, 0)
    ce_terms, z_terms = [], []
    dl = np.zeros((B, V))
    lse_all = np.empty(B)
    for r0 in range(0, B, row_block):
        r1 = min(B, r0 + row_block)
        rows = np.arange(r1 - r0)
        z = widen(x[r0:r1])
        L = lse(z)
        lse_all[r0:r1] = L
        v = valid[r0:r1]
        ce_terms.append(np.where(v, L - z[rows, y[r0:r1]], 0.0))
        z_terms.append(np.where(v, L * L, 0.0))
        d = np.exp(z - L[:, None]) * (1.0 + 2.0 * z_loss * L)[:, None]
        d[rows, y[r0:r1]] -= 1.0
        dl[r0:r1] = d * v[:, None]
    ce_sum = math.fsum(np.concatenate(ce_terms).tolist()) if ce_terms else 0.0
    z_sum = math.fsum(np.concatenate(z_terms).tolist()) if z_terms else 0.0
    return dict(ce_sum=ce_sum, z_sum=z_sum, n_valid=int(valid.sum()), lse=lse_all, dlogits=dl)


def ce_reference_loops(logits_, labels, ignore_index: int = -100, z_loss: float = 0.0) -> dict:
    """Element-by-element version of ``ce_reference`` for tiny inputs."""
    x = widen(logits_)
    B, V = x.shape
    ce_sum, z_sum, n_valid = [], [], 0
    D = np.zeros((B, V))
    for i in range(B):
        y = int(labels[i])
        if y == ignore_index or not (0 <= y < V):
            continue
        n_valid += 1
        row = [float(v) for v in x[i]]
        m = max(row)
        L = m + math.log(math.fsum(math.exp(v - m) for v in row))
        ce_sum.append(L - row[y])
        z_sum.append(L * L)
        for j in range(V):
            D[i, j] = math.exp(row[j] - L) * (1.0 + 2.0 * z_loss * L) - (1.0 if j == y else 0.0)
    return dict(ce_sum=math.fsum(ce_sum), z_sum=math.fsum(z_sum), n_valid=n_valid, dlogits=D)


def logit_avg(hidden, W, bias=None, row_block: int = 512) -> np.ndarray:
    """Average logit of every vocabulary entry over the batch, (1/BT) sum_t z[t, n] with z = hidden . W^T
    (+ b) (p2 "Forward pass": logit_avg, the mean logit per vocabulary entry, saved for the backward
    pass).  float64; the rows are summed block by block to bound memory."""
    h = widen(hidden)
    w = widen(W)
    b = None if bias is None else widen(bias)
    BT = h.shape[0]
    col_sum = np.zeros(w.shape[0])
    for r0 in range(0, BT, row_block):
        z = h[r0:r0 + row_block] @ w.T
        if b is not None:
            z += b[None, :]
        col_sum += z.sum(axis=0)
    if BT == 0:
        return col_sum + (b if b is not None else 0.0)
    return col_sum / BT


def vocab_order(avg) -> np.ndarray:
    """The vocabulary sorted by average logit, largest first (p2 "Vocabulary Sorting"): entry k of the
    result is the vocabulary index placed at sorted position k.  Equal keys keep increasing index
    order."""
    a = np.asarray(avg, dtype=np.float64)
    return np.argsort(-a, kind="stable").astype(np.int64)
