"""Partition of a prefill across ranks (one GPU each) by independent work units.

A unit is one (batch row b, KV head h_kv) pair: the query heads h_kv * g .. h_kv * g + g - 1 (g = Hq / Hkv)
attend to that KV head only, and a unit's BlockMask rows are those of its batch row and heads. Units
share nothing on the hot path, so ranks need no collective: each builds its own mask for its units and
runs the forward on its own slices of Q, K, V, O and LSE.

Units are numbered KV-head-major, u = h_kv * B + b, and rank r owns the contiguous range
[r * n / world, (r + 1) * n / world) of the n = B * Hkv units. A range is at most three rectangles
(batch rows b0 .. b1 x KV heads h0 .. h1): a partial KV head at each end and whole KV heads between. Each
rectangle is one local problem of b1 - b0 batch rows, (h1 - h0) * g query heads and h1 - h0 KV heads,
whose per-head parameters (ALiBi slopes, relative-bias rows) and per-batch state (document ids, query
offsets) are the matching slices of the global ones.

This module slices data only; it holds none of the method's arithmetic.
"""
from __future__ import annotations

from typing import List, Tuple

import numpy as np

from . import synth
from .workloads import TID_K, TID_Q, TID_V, Prefill

Piece = Tuple[int, int, int, int]  # (b0, b1, h0, h1): batch rows b0 .. b1 - 1, KV heads h0 .. h1 - 1


def unit_range(B: int, Hkv: int, world: int, rank: int) -> Tuple[int, int]:
    """The contiguous range of unit numbers (KV-head-major) that rank `rank` of `world` owns."""
    if not (B >= 1 and Hkv >= 1 and world >= 1 and 0 <= rank < world):
        raise ValueError("bad partition arguments")
    n = B * Hkv
    return rank * n // world, (rank + 1) * n // world


def pieces_for_rank(B: int, Hkv: int, world: int, rank: int) -> List[Piece]:
    """The rectangles (b0, b1, h0, h1) covering rank `rank`'s units, in unit order."""
    start, end = unit_range(B, Hkv, world, rank)
    pieces: List[Piece] = []
    u = start
    while u < end:
        hk, b = divmod(u, B)
        if b > 0 or end - u < B:                 # a part of one KV head's batch rows
            b1 = min(B, b + (end - u))
            pieces.append((b, b1, hk, hk + 1))
            u += b1 - b
        else:                                    # whole KV heads
            n_heads = (end - u) // B
            pieces.append((0, B, hk, hk + n_heads))
            u += n_heads * B
    return pieces


def units_of(pieces: List[Piece]) -> List[Tuple[int, int]]:
    """The (b, h_kv) units the rectangles cover."""
    return [(b, h) for (b0, b1, h0, h1) in pieces for h in range(h0, h1) for b in range(b0, b1)]


def slice_prefill(w: Prefill, piece: Piece, q_offset=None):
    """The local problem of one rectangle: a Prefill of b1 - b0 batch rows and (h1 - h0) * g query heads
    whose inputs are the global ones' slices (taken from `w` if generated, else drawn directly from the
    counter-based generator at the global offsets), with the score rule's per-head arrays and the document
    ids sliced to match; and the query offsets of its batch rows (if `q_offset` is given)."""
    b0, b1, h0, h1 = piece
    g = w.Hq // w.Hkv
    qh0, qh1 = h0 * g, h1 * g
    loc = Prefill(f"{w.name}[b{b0}:{b1},kv{h0}:{h1}]", b1 - b0, qh1 - qh0, h1 - h0, w.q_len, w.kv_len, w.d, w.bq,
                  w.bk, list(w.rule), dict(w.score), w.scale, w.seed, doc_lens=w.doc_lens)
    if w.q_bits is not None:
        loc.q_bits = np.ascontiguousarray(w.q_bits[b0:b1, qh0:qh1])
        loc.k_bits = np.ascontiguousarray(w.k_bits[b0:b1, h0:h1])
        loc.v_bits = np.ascontiguousarray(w.v_bits[b0:b1, h0:h1])
    else:
        def draw(tid, H, h_lo, h_hi, n):
            rows = [synth.normal_bf16_bits(w.seed, tid, (h_hi - h_lo, n, w.d), first=((b * H + h_lo) * n) * w.d)
                    for b in range(b0, b1)]
            return np.ascontiguousarray(np.stack(rows))
        loc.q_bits = draw(TID_Q, w.Hq, qh0, qh1, w.q_len)
        loc.k_bits = draw(TID_K, w.Hkv, h0, h1, w.kv_len)
        loc.v_bits = draw(TID_V, w.Hkv, h0, h1, w.kv_len)
    if w.doc_ids is not None:
        loc.doc_ids = w.doc_ids if w.doc_ids.shape[0] == 1 else np.ascontiguousarray(w.doc_ids[b0:b1])
    for key in ("alibi_slopes", "rel_bias"):
        if w.score.get(key) is not None:
            loc.score[key] = np.ascontiguousarray(np.asarray(w.score[key])[qh0:qh1])
    off = None if q_offset is None else np.ascontiguousarray(np.asarray(q_offset)[b0:b1])
    return loc, off
