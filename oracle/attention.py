"""Textbook softmax decode attention over reconstructed keys and values (float64).

[TQ-KV] "Marco Teórico" (K-V asymmetry): keys enter attention through inner
products with the query, values through an attention-weighted sum.
[HEADQ] "Espaço de Pontuação da Chave": the score of key j is q^T k_j / sqrt(d),
and "Geometria de Leitura de Valores": the readout is sum_j p_j v_j.

Grouped query heads: query head h reads KV head floor(h / G), G = H_q / H_kv.
A sequence of length 0 has no keys; its output is defined as 0.
"""

import numpy as np


def softmax(s):
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


def decode_attention(q, K, V):
    """One query vector q (d), keys K (T x d), values V (T x d) -> output (d)."""
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    d = q.shape[-1]
    p = softmax(K @ q / np.sqrt(d))
    return p @ V


def decode_attention_gqa(q, K, V, seq_len):
    """q: (B, H_q, d); K, V: (B, H_kv, >=T, d); seq_len: (B,) -> (B, H_q, d)."""
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        T = int(seq_len[b])
        for h in range(Hq):
            out[b, h] = decode_attention(q[b, h], K[b, h // G, :T], V[b, h // G, :T])
    return out


def logits(q, K):
    """Scores q^T k_j / sqrt(d) for all keys j."""
    return K @ q / np.sqrt(q.shape[-1])
