"""CPU oracle for pack -> bidirectional ragged attention -> unpack (fp64, numpy).

TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
benchmark's CPU-baseline / reference arm may import or run this module; the
product path never does, and this module imports nothing from the CUDA path.

What it follows.  "Dispatch-Aware Ragged Attention for Pruned Vision
Transformers" (arXiv 2604.15408), abstract (both revisions), and the
agents-report.net article on it ("Triton Ragged Attention 與
pack-attend-unpack ..."), section "方法概覽：pack-attend-unpack 流程"
(method overview), whose three bullets are the three steps below:

  1. fused token packing: from the per-image pruning decision, index work
     produces per-image offsets (``cu_seqlens``) and destination indices, and
     the surviving tokens are copied into one flat buffer;
  2. bidirectional ragged attention computed directly on that compact buffer;
  3. unpack: results go back to their original positions in the batch tensor
     using ``cu_seqlens``.

The abstract states that the packed result reproduces padded SDPA (the same
predictions, logits within a small bound), i.e. the method computes exact
softmax attention restricted to each image's kept tokens.  This oracle is that
plain definition written out, step by step, with no blocking or fusion.

Readings where the pages say nothing (each is listed in the design notes):
  * any nonzero mask byte means "keep";
  * packed order is images in batch order, tokens in their original order;
  * non-causal attention among the image's own kept tokens only;
  * softmax scale is a parameter (1/sqrt(64) for ViT heads);
  * pruned output positions are written as zeros;
  * an image with no kept token contributes no rows and an all-zero output.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(brute force over all masks of tiny sizes, torch fp64 SDPA on the padded
tensor, closed forms, invariants, and an exact sympy evaluation).
"""
from __future__ import annotations

import math

import numpy as np


def pack_indices(keep):
    """Step 1 index work: (cu_seqlens [B+1], dst_idx [B*N], src_idx [T]) as int32.

    cu_seqlens[b] is the number of kept tokens in images before b;
    dst_idx[b*N + j] is the packed row of token (b, j), or -1 if pruned;
    src_idx[t] is the flat padded position b*N + j of packed row t.
    """
    keep = np.asarray(keep)
    B, N = keep.shape
    cu_seqlens = np.zeros(B + 1, dtype=np.int32)
    dst_idx = np.full(B * N, -1, dtype=np.int32)
    src_idx = []
    t = 0
    for b in range(B):
        cu_seqlens[b] = t
        for j in range(N):
            if keep[b, j] != 0:
                dst_idx[b * N + j] = t
                src_idx.append(b * N + j)
                t += 1
    cu_seqlens[B] = t
    return cu_seqlens, dst_idx, np.asarray(src_idx, dtype=np.int32)


def pack_rows(x, src_idx):
    """Step 1 copy: packed[t] = x[b, j] for src_idx[t] = b*N + j (bit copy, any dtype)."""
    x = np.asarray(x)
    B, N = x.shape[:2]
    flat = x.reshape((B * N,) + x.shape[2:])
    out = np.empty((len(src_idx),) + x.shape[2:], dtype=x.dtype)
    for t, s in enumerate(src_idx):
        out[t] = flat[s]
    return out


def attend(qp, kp, vp, cu_seqlens, scale):
    """Step 2: O[t] for every packed row, fp64.

    For image b (rows cu[b]..cu[b+1]-1) and head h:
        S = scale * Q K^T,  P = exp(S - rowmax(S)) / rowsum,  O = P V,
    with no causal mask and only the image's own kept tokens as keys.
    ``qp``, ``kp``, ``vp`` are [T, H, d] arrays already holding the exact
    values of the low-precision inputs.
    """
    qp = np.asarray(qp, dtype=np.float64)
    kp = np.asarray(kp, dtype=np.float64)
    vp = np.asarray(vp, dtype=np.float64)
    T, H, d = qp.shape
    out = np.zeros((T, H, d), dtype=np.float64)
    B = len(cu_seqlens) - 1
    for b in range(B):
        s0, s1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if s1 <= s0:
            continue
        for h in range(H):
            Q = qp[s0:s1, h, :]
            K = kp[s0:s1, h, :]
            V = vp[s0:s1, h, :]
            S = scale * (Q @ K.T)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P = P / P.sum(axis=1, keepdims=True)
            out[s0:s1, h, :] = P @ V
    return out


def attend_row(qp, kp, vp, cu_seqlens, scale, t, h):
    """One output row O[t, h, :] of ``attend`` (for sampled checks at large sizes)."""
    B = len(cu_seqlens) - 1
    b = int(np.searchsorted(np.asarray(cu_seqlens), t, side="right")) - 1
    assert 0 <= b < B and cu_seqlens[b] <= t < cu_seqlens[b + 1]
    s0, s1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
    q = np.asarray(qp[t, h, :], dtype=np.float64)
    K = np.asarray(kp[s0:s1, h, :], dtype=np.float64)
    V = np.asarray(vp[s0:s1, h, :], dtype=np.float64)
    s = scale * (K @ q)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ V


def unpack(op, dst_idx, B, N):
    """Step 3: out[b, j] = O[dst_idx[b*N + j]] if kept, else zeros."""
    op = np.asarray(op)
    out = np.zeros((B * N,) + op.shape[1:], dtype=op.dtype)
    for x in range(B * N):
        t = int(dst_idx[x])
        if t >= 0:
            out[x] = op[t]
    return out.reshape((B, N) + op.shape[1:])


def pipeline(keep, q, k, v, scale):
    """Whole path on padded [B, N, H, d] fp64 inputs: returns (out, cu, dst, src)."""
    keep = np.asarray(keep)
    B, N = keep.shape
    cu, dst, src = pack_indices(keep)
    qp = pack_rows(np.asarray(q, dtype=np.float64), src)
    kp = pack_rows(np.asarray(k, dtype=np.float64), src)
    vp = pack_rows(np.asarray(v, dtype=np.float64), src)
    op = attend(qp, kp, vp, cu, scale)
    return unpack(op, dst, B, N), cu, dst, src


# ----------------------------------------------------------------------------
# The step before the path: a token-pruning decision made on the device.
#
# The abstract (both revisions) names EViT among the pruners the pipeline
# serves; the pages do not describe its rule.  The reading taken here is the
# plainest one consistent with "keep the tokens the class token attends to":
#   * an image's class token is its first kept token (position 0 in the
#     configurations, which always keep it);
#   * a kept token's score is the class token's softmax attention weight on
#     it, averaged over the heads;
#   * a pruning step keeps the class token and the top ceil(m * num / den)
#     of the image's m other kept tokens by score, equal scores going to the
#     lower position (a NaN score counts as -inf).


def cls_scores(qp, kp, cu_seqlens, src_idx, N, scale):
    """[B, N] fp64: for image b, the attention weights of its first kept token
    (packed row cu[b]) over the image's kept tokens, averaged over heads, at
    the tokens' original positions; 0 at positions with no kept token."""
    qp = np.asarray(qp, dtype=np.float64)
    kp = np.asarray(kp, dtype=np.float64)
    T, H, d = qp.shape
    B = len(cu_seqlens) - 1
    out = np.zeros((B, N), dtype=np.float64)
    for b in range(B):
        s0, s1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if s1 <= s0:
            continue
        acc = np.zeros(s1 - s0, dtype=np.float64)
        for h in range(H):
            s = scale * (kp[s0:s1, h, :] @ qp[s0, h, :])
            p = np.exp(s - s.max())
            acc += p / p.sum()
        for t in range(s0, s1):
            out[b, int(src_idx[t]) - b * N] = acc[t - s0] / H
    return out


def cls_weights(qp, kp, cu_seqlens, scale):
    """Per head, before the mean: a list over images b of fp64 [H, n_b]
    arrays, entry [h, i] the softmax weight (scale * <q, k> over the image's
    rows, head h) of the image's first row on its row i (packed order).
    Empty images give [H, 0] arrays."""
    qp = np.asarray(qp, dtype=np.float64)
    kp = np.asarray(kp, dtype=np.float64)
    T, H, d = qp.shape
    B = len(cu_seqlens) - 1
    out = []
    for b in range(B):
        s0, s1 = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        w = np.zeros((H, max(s1 - s0, 0)), dtype=np.float64)
        for h in range(H):
            if s1 <= s0:
                break
            s = scale * (kp[s0:s1, h, :] @ qp[s0, h, :])
            p = np.exp(s - s.max())
            w[h] = p / p.sum()
        out.append(w)
    return out


def topk_keep(scores, keep_prev, num, den):
    """[B, N] uint8: each image's first kept token plus the top
    ceil(m * num / den) of its m other kept tokens by score (descending,
    equal scores to the lower position, a NaN score counting as -inf)."""
    scores = np.asarray(scores, dtype=np.float64)
    keep_prev = np.asarray(keep_prev)
    B, N = keep_prev.shape
    out = np.zeros((B, N), dtype=np.uint8)
    for b in range(B):
        kept = [j for j in range(N) if keep_prev[b, j] != 0]
        if not kept:
            continue
        out[b, kept[0]] = 1
        others = kept[1:]
        m = len(others)
        k = (m * num + den - 1) // den
        key = lambda j: (-(scores[b, j]) if scores[b, j] == scores[b, j] else math.inf, j)   # NaN -> -inf
        for j in sorted(others, key=key)[:k]:
            out[b, j] = 1
    return out


# ----------------------------------------------------------------------------
# The rest of a ViT block on the compact buffer: a linear layer over the
# packed rows only (the article's problem section: padding wastes masked
# multiplies; packing removes them from every layer, not only attention).


def linear_packed(a, w, bias, T):
    """fp64 [T, N]: rows t < T of the packed [cap, K] matrix a times w^T
    ([N, K], the nn.Linear layout), plus bias [N] when given."""
    a = np.asarray(a, dtype=np.float64)[: int(T)]
    w = np.asarray(w, dtype=np.float64)
    out = a @ w.T
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)[None, :]
    return out
