"""Independent numpy fp64 restatement of the attention definition.

TEST INFRASTRUCTURE, used only to cross-check the C oracle on small inputs.
It is written vectorised (whole score matrix at once) so that it shares no
structure with the row loops of oracle.c. Definition: "Warmup Guide —
Inference Optimization at Depth", Chapters 1, 2 and 4 (S = Q K^T / sqrt(d),
safe softmax, O = P V), with the causal reading j <= i + (Sk - Sq).
"""
from __future__ import annotations

import numpy as np
import torch


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def attention_np(q, k, v, causal: bool, scale: float):
    """q [..., Sq, d], k/v [..., Sk, d] as float64 arrays -> (o, lse)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    sc = float(np.float32(scale))
    s = sc * np.einsum("...id,...jd->...ij", q, k)
    Sq, Sk = s.shape[-2], s.shape[-1]
    if causal:
        i = np.arange(Sq)[:, None]
        j = np.arange(Sk)[None, :]
        hidden = j > i + (Sk - Sq)
        s = np.where(hidden, -np.inf, s)
    m = s.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe)
    l = e.sum(axis=-1, keepdims=True)
    p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    o = p @ v
    with np.errstate(divide="ignore"):
        lse = np.where(empty[..., 0], -np.inf, (m_safe + np.log(np.where(l > 0, l, 1.0)))[..., 0])
    return o, lse
