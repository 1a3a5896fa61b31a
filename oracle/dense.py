"""Dense NumPy fp64 brute force of the same attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY.  An independent second statement of the definition
used to pin the C oracle: each request's K and V are materialised as whole
matrices by NumPy indexing of the HND pool, then the masked score matrix
S = Q K^T * sm_scale is built in full, softmax is taken row-wise and multiplied
by V ("Chunked prefill" (k4i.top), #correctness: token i sees positions j <= i;
"Disaggregated prefill and decode" (Perplexity), "Sharded KV cache transfers":
HND puts heads before tokens inside a page).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def request_kv(pool_bits: np.ndarray, page_ids: np.ndarray, kv_len: int):
    """K, V of one request as [kv_len, Hkv, d] fp64 from the HND pool."""
    pages = bf16_bits_to_f64(pool_bits[np.asarray(page_ids, np.int64)])  # [np, 2, Hkv, P, d]
    n, _, Hkv, P, d = pages.shape
    # [np, kv, Hkv, P, d] -> [kv, np, P, Hkv, d] -> [kv, np*P, Hkv, d]
    tok = pages.transpose(1, 0, 3, 2, 4).reshape(2, n * P, Hkv, d)
    return tok[0, :kv_len], tok[1, :kv_len]


def attention(q_bits, pool_bits, qo_indptr, kv_indptr, page_indices, last_page_len,
              causal, sm_scale, num_qo_heads, tree_mask=None):
    """(out [nnz, Hq, d], lse [nnz, Hq], weights: list per request [Hq, qo, kv]).

    tree_mask: optional uint32 [nnz, words] rows ("Accelerating Sonar through
    speculation", EAGLE: tree verification under a custom mask): the allowed
    matrix of a request is all cached columns, plus, over its new-token
    columns, the lower triangle of the unpacked mask bits with the diagonal."""
    q = bf16_bits_to_f64(q_bits)
    P = pool_bits.shape[3]
    Hkv = pool_bits.shape[2]
    g = num_qo_heads // Hkv
    outs, lses, ws = [], [], []
    for r in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[r]), int(qo_indptr[r + 1])
        p0, p1 = int(kv_indptr[r]), int(kv_indptr[r + 1])
        kv_len = 0 if p1 == p0 else (p1 - p0 - 1) * P + int(last_page_len[r])
        qo = q1 - q0
        if qo == 0:
            ws.append(None)
            continue
        K, V = request_kv(pool_bits, page_indices[p0:p1], kv_len)
        K = np.repeat(K, g, axis=1)  # [kv, Hq, d]: head h reads kv head h // g
        V = np.repeat(V, g, axis=1)
        Q = q[q0:q1]  # [qo, Hq, d]
        S = np.einsum("ihc,jhc->hij", Q, K) * sm_scale  # [Hq, qo, kv]
        if causal:
            i = np.arange(qo)[:, None]
            j = np.arange(kv_len)[None, :]
            allowed = j <= (kv_len - qo) + i
            if tree_mask is not None:
                bits = np.unpackbits(np.ascontiguousarray(tree_mask[q0:q1]).view(np.uint8), axis=1,
                                     bitorder="little")[:, :qo].astype(bool)
                new = np.tril(bits, -1) | np.eye(qo, dtype=bool)
                allowed = np.concatenate([np.ones((qo, kv_len - qo), bool), new], axis=1)
            S = np.where(allowed, S, -np.inf)
        m = S.max(axis=2, keepdims=True)
        E = np.exp(S - m)
        Z = E.sum(axis=2, keepdims=True)
        W = E / Z
        O = np.einsum("hij,jhc->ihc", W, V)
        outs.append(O)
        lses.append((m[..., 0] + np.log(Z[..., 0])).T)
        ws.append(W)
    d = pool_bits.shape[4]
    out = np.concatenate(outs, 0) if outs else np.zeros((0, num_qo_heads, d))
    lse = np.concatenate(lses, 0) if lses else np.zeros((0, num_qo_heads))
    return out, lse, ws
