"""Pure-Python brute force for tiny attention cases (fp64, contiguous K/V).

TEST INFRASTRUCTURE ONLY.  Independent of ``ref.c``: no paging at all, just
the definition of causal attention with new tokens at the end of each
sequence, as in the KV-cache toy of the inference-system notes ("推理系统",
CS 与 LLM 学习知识库): new token i of T sees the first S - T + i + 1 keys.
Grouped heads: query head h uses KV head h // (Hq // Hkv).
"""
from __future__ import annotations

import math


def attention(q, k, v, scale):
    """q: [T][Hq][D], k/v: [S][Hkv][D] nested lists of floats (one sequence).

    Returns [T][Hq][D] as nested lists.
    """
    t_len, s_len = len(q), len(k)
    hq, hkv = len(q[0]), len(k[0])
    group = hq // hkv
    out = []
    for i in range(t_len):
        visible = s_len - t_len + i + 1
        rows = []
        for h in range(hq):
            g = h // group
            scores = []
            for j in range(visible):
                scores.append(scale * sum(a * b for a, b in zip(q[i][h], k[j][g])))
            m = max(scores)
            w = [math.exp(x - m) for x in scores]
            z = sum(w)
            dim = len(v[0][g])
            rows.append([sum(w[j] * v[j][g][d] for j in range(visible)) / z for d in range(dim)])
        out.append(rows)
    return out
