"""Seeded synthetic inputs for the attention-forward workloads.

This module holds shapes and random draws only; none of the attention
arithmetic lives here. Both the CUDA path and the fp64 oracle are fed from
these generators, so both see the same bf16 bits.

Recipe (every workload): one CPU ``torch.Generator`` seeded with the
workload's seed draws Q, then K, then V, in that order. Each draw is iid
N(0, 1) in fp32, multiplied by the workload's factor (1 except for Q in the
stress variant), then rounded to bf16. The softmax scale is 1/sqrt(d),
rounded to fp32 — the scale of "Warmup Guide — Inference Optimization at
Depth", Chapter 4.

The shapes are the pages' own workloads:
  * the [B, H, S, S] score matrix example at B=4, H=32, S=8192
    ("FlashAttention, speculative decoding, quantisation and parallelism",
    "The problem it solves");
  * the 32K-token score matrix example ("Warmup Guide", Chapter 1);
  * the speculative-decoding verify step, where the target scores k+1
    positions in one forward pass over a KV cache (page 1, "Speculative
    decoding"; "Lecture 06", section 5, Flash-Decoding).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    seed: int
    q_factor: float = 1.0

    @property
    def scale(self) -> float:
        """1/sqrt(d) rounded to fp32, returned as the Python float of that fp32."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    @property
    def q_shape(self):
        return (self.B, self.H, self.Sq, self.d)

    @property
    def kv_shape(self):
        return (self.B, self.H, self.Sk, self.d)

    def visible_keys(self, i: int) -> int:
        """Number of keys query row i may attend to (bottom-right causal alignment)."""
        if not self.causal:
            return self.Sk
        return max(0, min(self.Sk, i + (self.Sk - self.Sq) + 1))

    def visible_pairs(self) -> int:
        """Exact count of (query, key) pairs that enter the softmax, per (b, h)."""
        if not self.causal:
            return self.Sq * self.Sk
        off = self.Sk - self.Sq
        total = 0
        # closed form of sum_i clamp(i + off + 1, 0, Sk) without a Python loop
        # over long sequences: split at the rows where clamping switches.
        lo = max(0, -off)                      # first row with >= 1 visible key
        hi = min(self.Sq, self.Sk - off - 1)   # first row that sees all Sk keys
        if hi > lo:
            a, b = lo + off + 1, hi - 1 + off + 1
            total += (a + b) * (hi - lo) // 2
        total += max(0, self.Sq - max(hi, lo)) * self.Sk
        return total

    def exact_flops(self) -> int:
        """Algorithmic FLOPs: 2*d for QK^T plus 2*d for PV per visible pair."""
        return 4 * self.d * self.visible_pairs() * self.B * self.H

    def fa_convention_flops(self) -> int:
        """4*B*H*Sq*Sk*d, halved when causal (the usual FlashAttention count)."""
        f = 4 * self.B * self.H * self.Sq * self.Sk * self.d
        return f // 2 if self.causal else f

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once (bf16), write O (bf16) and LSE (fp32)."""
        q = self.B * self.H * self.Sq * self.d * 2
        kv = 2 * self.B * self.H * self.Sk * self.d * 2
        o = q
        lse = self.B * self.H * self.Sq * 4
        return q + kv + o + lse

    def score_matrix_bytes(self, elem_bytes: int = 2) -> int:
        """Size of the materialised [B, H, Sq, Sk] score matrix that the tiled path avoids."""
        return self.B * self.H * self.Sq * self.Sk * elem_bytes


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_b1h1s256d64_noncausal", 1, 1, 256, 256, 64, False, 0),
        Workload("tiny_b1h1s256d64_causal", 1, 1, 256, 256, 64, True, 0),
        Workload("prefill_b4h32s2048d128_causal", 4, 32, 2048, 2048, 128, True, 1),
        Workload("prefill_b4h32s2048d128_causal_q4", 4, 32, 2048, 2048, 128, True, 1, 4.0),
        Workload("prefill_b4h32s8192d128_causal", 4, 32, 8192, 8192, 128, True, 2),
        Workload("prefill_b1h32s32768d64_causal", 1, 32, 32768, 32768, 64, True, 3),
        Workload("verify_b16h32q5k4096d128", 16, 32, 5, 4096, 128, True, 4),
    ]
}

# The headline workload: causal prefill at B=4, H=32, S=8192, d=128.
HEADLINE = "prefill_b4h32s8192d128_causal"
VERIFY = "verify_b16h32q5k4096d128"


def custom(B, H, Sq, Sk, d, causal, seed=0, q_factor=1.0, name=None) -> Workload:
    return Workload(name or f"custom_b{B}h{H}q{Sq}k{Sk}d{d}{'c' if causal else 'n'}",
                    B, H, Sq, Sk, d, bool(causal), seed, q_factor)


def make_qkv(w: Workload, device="cpu"):
    """Draw Q, K, V for workload ``w`` (bf16, contiguous [B, H, S, d])."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(w.q_shape, generator=g, dtype=torch.float32)
    if w.q_factor != 1.0:
        q.mul_(w.q_factor)
    q = q.to(torch.bfloat16)
    k = torch.randn(w.kv_shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(w.kv_shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def make_qkv_device(w: Workload, device="cuda"):
    """Q, K, V for workload ``w`` drawn on ``device`` by a seeded device
    generator, for shapes too large to draw on the host (tensors past 2^31
    elements). Same recipe as ``make_qkv`` (iid N(0, 1) in fp32, Q times
    q_factor, cast to bf16), drawn in slices of the batch dimension of about
    2^27 elements; the values differ from ``make_qkv``'s for the same seed."""
    g = torch.Generator(device=device).manual_seed(w.seed)
    out = []
    for shape, factor in ((w.q_shape, w.q_factor), (w.kv_shape, 1.0), (w.kv_shape, 1.0)):
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        per_b = shape[1] * shape[2] * shape[3]
        step = max(1, (1 << 27) // per_b)
        for b0 in range(0, shape[0], step):
            b1 = min(shape[0], b0 + step)
            x = torch.randn((b1 - b0,) + tuple(shape[1:]), generator=g, dtype=torch.float32,
                            device=device)
            if factor != 1.0:
                x.mul_(factor)
            t[b0:b1].copy_(x)
            del x
        out.append(t)
    return tuple(out)


def make_qkv_fp8(w: Workload, device="cpu"):
    """E4M3 inputs for workload ``w``: the same N(0, 1) draws as ``make_qkv``
    (seed, order, q_factor), each tensor divided by a power-of-two descale
    2^ceil(log2(amax / 448)) so that it fits E4M3's range without clamping, then
    cast by torch (round to nearest even). Returns (q8, k8, v8, descales), with
    q8/k8/v8 torch.float8_e4m3fn [B, H, S, d] and descales = (dq, dk, dv) floats:
    an input byte stands for descale * its E4M3 value."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(w.q_shape, generator=g, dtype=torch.float32)
    if w.q_factor != 1.0:
        q.mul_(w.q_factor)
    k = torch.randn(w.kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(w.kv_shape, generator=g, dtype=torch.float32)
    out, descales = [], []
    for t in (q, k, v):
        amax = float(t.abs().max()) if t.numel() else 1.0
        ds = 2.0 ** math.ceil(math.log2(max(amax, 1e-30) / 448.0))
        out.append((t / ds).to(torch.float8_e4m3fn))
        descales.append(ds)
    if device != "cpu":
        out = [t.to(device) for t in out]
    return out[0], out[1], out[2], tuple(descales)


def sample_rows(w: Workload, per_head: int | None = None, n_total: int | None = None,
                seed: int = 12345, tile: int = 128):
    """Seeded (b, h, i) query rows for sampled parity checks at full size.

    Always includes the first and last row and the rows on either side of
    query-tile boundaries (127/128, 255/256, ...), the two classic bug sites
    the pages name ("Warmup Guide", Lab Walkthrough: non-divisible tile
    boundaries and the causal diagonal blocks).
    """
    g = torch.Generator().manual_seed(seed)
    special = sorted({0, w.Sq - 1, min(tile - 1, w.Sq - 1), min(tile, w.Sq - 1),
                      min(2 * tile - 1, w.Sq - 1), min(2 * tile, w.Sq - 1),
                      max(0, w.Sq - tile), max(0, w.Sq - tile - 1)})
    rows = []
    if per_head is not None:
        for b in range(w.B):
            for h in range(w.H):
                extra = torch.randint(0, w.Sq, (max(0, per_head - len(special)),), generator=g)
                for i in special + extra.tolist():
                    rows.append((b, h, int(i)))
    else:
        n_total = n_total or 64
        bh = torch.randint(0, w.B * w.H, (n_total,), generator=g).tolist()
        ii = torch.randint(0, w.Sq, (n_total,), generator=g).tolist()
        for n, i in enumerate(special):
            ii[n % n_total] = i
        rows = [(x // w.H, x % w.H, int(i)) for x, i in zip(bh, ii)]
    return rows


def with_seed(w: Workload, seed: int) -> Workload:
    return replace(w, seed=seed)


def make_tree_masks(B: int, Sq: int, seed: int = 0):
    """Seeded random draft trees, one per sequence, as uint32 [B, Sq] masks.

    Candidate 0 is the root; candidate i > 0 hangs under a random earlier
    candidate. Bit k of mask[b][i] is set when candidate k is an ancestor of
    candidate i or i itself (what tree-attention lets it see among the drafts).
    """
    g = torch.Generator().manual_seed(seed)
    masks = torch.zeros((B, Sq), dtype=torch.int64)
    for b in range(B):
        for i in range(Sq):
            parent = int(torch.randint(0, i, (1,), generator=g)) if i > 0 else -1
            masks[b, i] = (1 << i) | (int(masks[b, parent]) if parent >= 0 else 0)
    return masks.to(torch.int32)   # bit patterns; Sq <= 31


def make_paged_kv(k: torch.Tensor, v: torch.Tensor, seq_lens, page_size: int,
                  extra_pages: int = 3, seed: int = 0):
    """Scatter contiguous K, V [B, H, Sk, d] into page pools [num_pages, H, page_size, d]
    through a seeded random block table. Keys past seq_lens[b] are not stored.
    Returns (k_pages, v_pages, block_table int32 [B, max_pages], seq_lens int32 [B])."""
    B, H, Sk, d = k.shape
    max_pages = -(-Sk // page_size)
    need = sum(-(-int(n) // page_size) for n in seq_lens)
    num_pages = need + extra_pages
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(num_pages, generator=g)
    k_pages = torch.randn((num_pages, H, page_size, d), generator=g).to(k.dtype)
    v_pages = torch.randn((num_pages, H, page_size, d), generator=g).to(v.dtype)
    table = torch.full((B, max_pages), -7, dtype=torch.int32)   # unused entries: garbage
    nxt = 0
    for b in range(B):
        for lp in range(-(-int(seq_lens[b]) // page_size)):
            phys = int(order[nxt])
            nxt += 1
            table[b, lp] = phys
            lo, hi = lp * page_size, min((lp + 1) * page_size, int(seq_lens[b]))
            k_pages[phys, :, : hi - lo] = k[b, :, lo:hi]
            v_pages[phys, :, : hi - lo] = v[b, :, lo:hi]
    return k_pages, v_pages, table, torch.tensor(list(seq_lens), dtype=torch.int32)

