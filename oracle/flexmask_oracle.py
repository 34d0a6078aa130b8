"""Plain, slow fp64 CPU oracle for masked attention over a BlockMask.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg
may import this module. It shares no code with the CUDA path: its own rule evaluator, its own block
classification and compaction, its own softmax. It reads rules as plain data (see workloads.py for the spec).

Sources (web pages on FlexAttention / FlashAttention; titles as printed):
  [FX]  "5.1.2 FlexAttention: from rules to fused kernels" (PaperTrace)
  [FC]  "FlexAttention: compiler optimisation of custom attention"
  [K5]  "5 Kernels: turning logical sparsity into real speed-ups" (PaperTrace)
  [FA]  FlashAttention self-test answers (LLM tutorial, L24)
  [CP]  article on causal block-level geometric pruning

What the oracle computes (exact attention restricted to the mask, [FA] Q8; [FX] 6.3):
  A(b,h,i,j) = rule(b,h,i_g,j) and i < Q_LEN and j < KV_LEN,   i_g = i + q_offset[b]    ([FC] section 6)
  s_ij = scale * <q_i, k_j>   (fp64 over the exact bf16 input values; scale defaults to 1/sqrt(d))
  s_ij <- softcap(s_ij + alibi + relbias)     fixed order c(a*s + r)                    ([FX] 1.2)
  s_ij <- -inf where not A                     (mask after score_mod)                  ([FX] 1.2, 3.1)
  two-pass softmax: m = max_j s_ij, l = sum_j e^(s_ij - m), O = sum_j e^(s_ij - m)/l * v_j, LSE = m + ln l
  empty row (m = -inf): O = 0, LSE = -inf                                              ([K5] section 3)
  document id of position t: doc_ids[b][t] for t in [0, doc_len), -1 outside, so a query position pushed
  past the id array by an offset shares a document only with keys whose id is -1       ([FX] 1.1 reading)
BlockMask tables ([FX] 2.1-2.2; [K5] section 4): per (b_m, h_m, query block r, KV block c) count the allowed
pairs over the full Bq x Bk footprint: 0 -> empty, Bq*Bk -> full, otherwise partial (pairs outside
[0,Q_LEN) x [0,KV_LEN) count as not allowed). Partial and full column lists per row, ascending, unused
slots 0; the query-side transpose per column, ascending.

Every function here is pinned by tests/test_oracle_pins.py against values the pages print, closed forms,
library routines (torch fp64 softmax / SDPA math path) and brute-force invariants. Parity unpinned: the
composition of a bias with the soft-cap beyond single-key closed forms, and rel-bias beyond tiny brute force.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

EMPTY, PARTIAL, FULL = 0, 1, 2


# ----------------------------------------------------------------------------------------------
# mask_mod: the allowed set ([FX] 1.1; [FC] section 2; prefix-LM as read from [CP] section 5)
# ----------------------------------------------------------------------------------------------
def rule_reads_doc(rule: Sequence[tuple]) -> bool:
    return any(op[0] == "doc" for op in rule)


def allowed(rule: Sequence[tuple], i_g: np.ndarray, j: np.ndarray,
            doc_q: Optional[np.ndarray] = None, doc_k: Optional[np.ndarray] = None) -> np.ndarray:
    """Evaluate a postfix mask rule on broadcastable integer arrays of global query positions i_g and KV
    positions j. doc_q / doc_k are the document ids at those positions (same broadcast shapes)."""
    shape = np.broadcast(i_g, j).shape
    stack = []
    for op in rule:
        name = op[0]
        if name == "true":
            stack.append(np.ones(shape, dtype=bool))
        elif name == "causal":                     # i >= j
            stack.append(np.broadcast_to(i_g >= j, shape))
        elif name == "window":                     # i - j < W (W includes the current token)
            stack.append(np.broadcast_to(i_g - j < int(op[1]), shape))
        elif name == "prefix":                     # j < P
            stack.append(np.broadcast_to(j < int(op[1]), shape))
        elif name == "doc":                        # d_b(i) == d_b(j)
            if doc_q is None or doc_k is None:
                raise ValueError("doc rule without document ids")
            stack.append(np.broadcast_to(doc_q == doc_k, shape))
        elif name in ("and", "or"):
            if len(stack) < 2:
                raise ValueError("malformed rule")
            b = stack.pop()
            a = stack.pop()
            stack.append((a & b) if name == "and" else (a | b))
        else:
            raise ValueError(f"unknown mask op {name!r}")
    if len(stack) != 1:
        raise ValueError("malformed rule")
    return np.asarray(stack[0], dtype=bool)


def _doc_at(doc_ids: Optional[np.ndarray], b: int, pos: np.ndarray) -> Optional[np.ndarray]:
    if doc_ids is None:
        return None
    row = doc_ids[b if doc_ids.shape[0] > 1 else 0]
    inside = (pos >= 0) & (pos < row.shape[0])
    out = np.full(pos.shape, -1, dtype=np.int64)
    out[inside] = row[pos[inside]]
    return out


def dense_allowed(rule, b: int, rows: np.ndarray, q_len: int, kv_len: int, q_offset: int = 0,
                  doc_ids: Optional[np.ndarray] = None, cols: Optional[np.ndarray] = None) -> np.ndarray:
    """A[i, j] for query indices `rows` (may run past q_len) and KV indices `cols` (default all kv_len)."""
    if cols is None:
        cols = np.arange(kv_len, dtype=np.int64)
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    i_g = i + int(q_offset)
    dq = _doc_at(doc_ids, b, i_g) if rule_reads_doc(rule) else None
    dk = _doc_at(doc_ids, b, j) if rule_reads_doc(rule) else None
    a = allowed(rule, i_g, j, dq, dk)
    return a & (i < q_len) & (j < kv_len) & (j >= 0)


# ----------------------------------------------------------------------------------------------
# BlockMask: classification, compaction and the query-side transpose ([FX] 2.1-2.2; [K5] 4)
# ----------------------------------------------------------------------------------------------
def block_mask(rule, B: int, H: int, q_len: int, kv_len: int, bq: int, bk: int,
               batch_dependent: bool = False, head_dependent: bool = False,
               q_offset: Optional[np.ndarray] = None, doc_ids: Optional[np.ndarray] = None,
               rows: Optional[Sequence[int]] = None) -> dict:
    """Return the BlockMask tables as int32 arrays (plus `block_class` uint8 [Bm,Hm,nq,nk]).

    Bm = B if batch_dependent else 1, Hm = H if head_dependent else 1 (FlexAttention's B=None / H=None
    broadcast). `rows`, if given, limits classification to those query block rows (others stay EMPTY and
    the transposes are then only valid for those rows)."""
    Bm = B if batch_dependent else 1
    Hm = H if head_dependent else 1
    nq = -(-q_len // bq)
    nk = -(-kv_len // bk)
    cls = np.zeros((Bm, Hm, nq, nk), dtype=np.uint8)
    cols = np.arange(nk * bk, dtype=np.int64)
    row_list = range(nq) if rows is None else rows
    for bm in range(Bm):
        off = 0 if q_offset is None else int(q_offset[bm])
        for hm in range(Hm):
            for r in row_list:
                qi = np.arange(r * bq, (r + 1) * bq, dtype=np.int64)
                a = dense_allowed(rule, bm, qi, q_len, kv_len, off, doc_ids, cols)   # [bq, nk*bk]
                cnt = a.reshape(bq, nk, bk).sum(axis=(0, 2))                          # pairs per block
                cls[bm, hm, r] = np.where(cnt == 0, EMPTY, np.where(cnt == bq * bk, FULL, PARTIAL))
    return tables_from_classes(cls, q_len, kv_len, bq, bk)


def tables_from_classes(cls: np.ndarray, q_len: int, kv_len: int, bq: int, bk: int) -> dict:
    Bm, Hm, nq, nk = cls.shape
    out = dict(Bm=Bm, Hm=Hm, q_len=q_len, kv_len=kv_len, bq=bq, bk=bk, nq=nq, nk=nk, block_class=cls)
    for name, want in (("kv", PARTIAL), ("full_kv", FULL)):
        num = np.zeros((Bm, Hm, nq), dtype=np.int32)
        idx = np.zeros((Bm, Hm, nq, nk), dtype=np.int32)
        for bm in range(Bm):
            for hm in range(Hm):
                for r in range(nq):
                    c = np.nonzero(cls[bm, hm, r] == want)[0]          # ascending column ids
                    num[bm, hm, r] = len(c)
                    idx[bm, hm, r, :len(c)] = c
        out[name + "_num"] = num
        out[name + "_idx"] = idx
    for name, want in (("q", PARTIAL), ("full_q", FULL)):
        num = np.zeros((Bm, Hm, nk), dtype=np.int32)
        idx = np.zeros((Bm, Hm, nk, nq), dtype=np.int32)
        for bm in range(Bm):
            for hm in range(Hm):
                for c in range(nk):
                    r = np.nonzero(cls[bm, hm, :, c] == want)[0]       # ascending row ids
                    num[bm, hm, c] = len(r)
                    idx[bm, hm, c, :len(r)] = r
        out[name + "_num"] = num
        out[name + "_idx"] = idx
    return out


def expand_tables(t: dict) -> np.ndarray:
    """M_hat: the element mask implied by the tables alone (full -> all true, partial -> marked 'partial',
    empty -> false). Returns int8 [Bm,Hm,nq*bq,nk*bk] with 0 empty, 1 partial, 2 full."""
    Bm, Hm, nq, nk, bq, bk = t["Bm"], t["Hm"], t["nq"], t["nk"], t["bq"], t["bk"]
    m = np.zeros((Bm, Hm, nq, nk), dtype=np.int8)
    for bm in range(Bm):
        for hm in range(Hm):
            for r in range(nq):
                for c in t["kv_idx"][bm, hm, r, :t["kv_num"][bm, hm, r]]:
                    m[bm, hm, r, c] = PARTIAL
                for c in t["full_kv_idx"][bm, hm, r, :t["full_kv_num"][bm, hm, r]]:
                    m[bm, hm, r, c] = FULL
    return np.repeat(np.repeat(m, bq, axis=2), bk, axis=3)


# ----------------------------------------------------------------------------------------------
# score_mod ([FX] 1.2): scaled score, then + ALiBi, + relative bias, then soft-cap, in that order
# ----------------------------------------------------------------------------------------------
def score_mod(s: np.ndarray, h: int, i_g: np.ndarray, j: np.ndarray, score: Optional[dict],
              kv_len: int) -> np.ndarray:
    if not score:
        return s
    dist = (np.asarray(i_g, dtype=np.int64) - np.asarray(j, dtype=np.int64)).astype(np.float64)
    slopes = score.get("alibi_slopes")
    if slopes is not None:
        s = s - float(slopes[h]) * dist                      # head-specific, distance-proportional bias
    rel = score.get("rel_bias")
    if rel is not None:
        delta = (np.asarray(i_g, dtype=np.int64) - np.asarray(j, dtype=np.int64)) + (kv_len - 1)
        delta = np.clip(delta, 0, 2 * kv_len - 2)
        s = s + np.asarray(rel, dtype=np.float64)[h][delta]  # r_h(i - j)
    c = float(score.get("softcap", 0.0) or 0.0)
    if c > 0.0:
        s = c * np.tanh(s / c)                               # c * tanh(s / c)
    return s


# ----------------------------------------------------------------------------------------------
# attention: the plain definition, two-pass softmax in fp64 ([FA] Q1, Q8; [FX] 3.1)
# ----------------------------------------------------------------------------------------------
def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, rule, rows: np.ndarray, b: int,
                   h: int, q_len: int, kv_len: int, scale: float, score: Optional[dict] = None,
                   q_offset: int = 0, doc_ids: Optional[np.ndarray] = None, return_p: bool = False,
                   bias_kv_len: Optional[int] = None):
    """Exact masked attention for the query rows `rows` of one (b, query head h).

    q_rows [n, d] fp64 (the query vectors of those rows), k/v [kv_len, d] fp64 (already the KV head
    floor(h/g)). Returns (O [n, d], LSE [n]) and optionally P [n, kv_len]. `bias_kv_len` is the KV_LEN the
    relative-bias table is laid out for (default kv_len)."""
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(kv_len, dtype=np.int64)
    a = dense_allowed(rule, b, rows, q_len, kv_len, q_offset, doc_ids)
    if not return_p:
        # A key that no row of this call may see contributes exactly zero to every row (its score becomes
        # -inf, e^-inf = 0: [FX] 1.2, [K5] 3), so its dot products are skipped; the rule was still
        # evaluated on every pair above.
        used = np.nonzero(a.any(axis=0))[0]
        if used.size < kv_len:
            j, a, k, v = j[used], a[:, used], k[used], v[used]
    s = scale * (q_rows @ k.T)
    s = score_mod(s, h, rows[:, None] + int(q_offset), j[None, :], score,
                  kv_len if bias_kv_len is None else bias_kv_len)
    s = np.where(a, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(len(rows), -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    p = np.exp(s - m_safe[:, None])                # exp(-inf) = 0 for masked pairs
    l = p.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    pn = p / l_safe[:, None]
    o = pn @ v
    o[empty] = 0.0
    lse = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    if return_p:
        return o, lse, pn
    return o, lse


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, rule, scale: Optional[float] = None,
              score: Optional[dict] = None, q_offset: Optional[np.ndarray] = None,
              doc_ids: Optional[np.ndarray] = None, rows: Optional[Sequence[int]] = None,
              heads: Optional[Sequence[tuple]] = None):
    """q [B,Hq,Q_LEN,d], k/v [B,Hkv,KV_LEN,d] (fp64). GQA: KV head = floor(h_q / g), g = Hq/Hkv, while the
    score rule reads the query head ([FX] 1.2, GQA paragraph). Returns O [B,Hq,n,d], LSE [B,Hq,n] for the
    query rows `rows` (default all) of every (b, h) in `heads` (default all; others left zero / -inf)."""
    B, Hq, q_len, d = q.shape
    Hkv, kv_len = k.shape[1], k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((B, Hq, len(rows), v.shape[-1]))
    lse = np.full((B, Hq, len(rows)), -np.inf)
    pairs = [(b, h) for b in range(B) for h in range(Hq)] if heads is None else heads
    for b, h in pairs:
        hk = h // g
        off = 0 if q_offset is None else int(q_offset[b])
        o[b, h], lse[b, h] = attention_rows(q[b, h, rows], k[b, hk], v[b, hk], rule, rows, b, h, q_len,
                                            kv_len, scale, score, off, doc_ids)
    return o, lse


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, rule,
                       scale: Optional[float] = None, score: Optional[dict] = None,
                       q_offset: Optional[np.ndarray] = None, doc_ids: Optional[np.ndarray] = None):
    """Gradients of the masked attention output O with respect to q, k, v for an upstream gradient dO
    ([FA] backward questions; [FX] 4.2): with s the scaled score, s' = score_mod(s) and P = softmax(s')
    over the allowed pairs,
        dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id,  dS' = P * (dP - D),
        dS = dS' * ds'/ds  (1 - (s'/c)^2 under the soft-cap c; biases do not depend on q or k),
        dQ = scale dS K,  dK = scale dS^T Q,
    summed over the query heads that share a KV head. Masked pairs and empty rows carry no gradient.
    q [B,Hq,Q_LEN,d], k/v [B,Hkv,KV_LEN,d], do like q (fp64). Returns dq, dk, dv (fp64)."""
    B, Hq, q_len, d = q.shape
    Hkv, kv_len = k.shape[1], k.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    rows = np.arange(q_len, dtype=np.int64)
    j = np.arange(kv_len, dtype=np.int64)
    c = float((score or {}).get("softcap", 0.0) or 0.0)
    for b in range(B):
        off = 0 if q_offset is None else int(q_offset[b])
        a = dense_allowed(rule, b, rows, q_len, kv_len, off, doc_ids)
        for h in range(Hq):
            hk = h // g
            s = scale * (q[b, h] @ k[b, hk].T)
            sm = score_mod(s, h, rows[:, None] + off, j[None, :], score, kv_len)
            o, _, p = attention_rows(q[b, h], k[b, hk], v[b, hk], rule, rows, b, h, q_len, kv_len, scale,
                                     score, off, doc_ids, return_p=True)
            dv[b, hk] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, hk].T
            delta = np.sum(do[b, h] * o, axis=1)
            ds = p * (dp - delta[:, None])
            if c > 0.0:
                ds = ds * (1.0 - (sm / c) ** 2)
            ds = np.where(a, ds, 0.0)
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def merge_partials(m: np.ndarray, l: np.ndarray, u: np.ndarray):
    """Merge split-softmax states ([K5] section 3): m = max_s m_s, l = sum_s e^(m_s - m) l_s,
    u = sum_s e^(m_s - m) u_s, O = u / l, LSE = m + ln l. Axis 0 indexes the splits; an empty split has
    m_s = -inf, l_s = 0, u_s = 0 and gets weight 0 ([FC] section 6)."""
    mm = np.max(m, axis=0)
    empty = ~np.isfinite(mm)
    mm_safe = np.where(empty, 0.0, mm)
    w = np.exp(m - mm_safe)                 # e^(-inf) = 0 for empty splits
    lt = np.sum(w * l, axis=0)
    ut = np.sum(w[..., None] * u, axis=0) if u.ndim == m.ndim + 1 else np.sum(w * u, axis=0)
    lt_safe = np.where(empty, 1.0, lt)
    o = ut / (lt_safe[..., None] if u.ndim == m.ndim + 1 else lt_safe)
    lse = np.where(empty, -np.inf, mm_safe + np.log(lt_safe))
    return o, lse


def split_state(s_row: np.ndarray, v: np.ndarray):
    """(m, l, u) of one key subset of a row: m = max s, l = sum e^(s-m), u = sum e^(s-m) v ([K5] 3)."""
    if s_row.size == 0 or not np.isfinite(s_row).any():
        return -np.inf, 0.0, np.zeros(v.shape[1])
    m = s_row.max()
    p = np.exp(s_row - m)
    return m, p.sum(), p @ v


# ----------------------------------------------------------------------------------------------
# paged decode ([FX] 5.1-5.2; [FC] section 6): logical KV position j lives in physical page
# page_table[b][j // page] at slot j % page; the rules use logical (global) positions.
# ----------------------------------------------------------------------------------------------
def gather_pages(pages: np.ndarray, page_table: np.ndarray, b: int, n_pages: int) -> np.ndarray:
    """Materialise request b's logical KV [Hkv, n_pages*page, d] from pages [P, Hkv, page, d]."""
    ids = page_table[b, :n_pages]
    if np.any(ids < 0) or np.any(ids >= pages.shape[0]):
        raise ValueError("page id out of range")
    sel = pages[ids]                                   # [n_pages, Hkv, page, d]
    return np.transpose(sel, (1, 0, 2, 3)).reshape(pages.shape[1], n_pages * pages.shape[2], pages.shape[3])


def decode_attention(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray, page_table: np.ndarray,
                     kv_lens: np.ndarray, rule, scale: Optional[float] = None, score: Optional[dict] = None,
                     doc_ids: Optional[np.ndarray] = None, requests: Optional[Sequence[int]] = None,
                     kv_len_table: Optional[int] = None):
    """One new token per request: q [Bz,Hq,d]; O [Bz,Hq,d], LSE [Bz,Hq]. Query position cur_pos = L_b - 1
    (global); KV positions beyond the request's materialised pages must be disallowed by the rule, which is
    checked here rather than assumed."""
    Bz, Hq, d = q.shape
    Hkv, page = k_pages.shape[1], k_pages.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros((Bz, Hq, d))
    lse = np.full((Bz, Hq), -np.inf)
    kv_len_table = kv_len_table if kv_len_table is not None else page_table.shape[1] * page
    for b in (range(Bz) if requests is None else requests):
        L = int(kv_lens[b])
        n_pages = -(-L // page)
        kb = gather_pages(k_pages, page_table, b, n_pages)
        vb = gather_pages(v_pages, page_table, b, n_pages)
        cur = L - 1
        beyond = np.arange(n_pages * page, kv_len_table, dtype=np.int64)
        if beyond.size and dense_allowed(rule, b, np.array([0]), 1, kv_len_table, cur, doc_ids, beyond).any():
            raise ValueError("rule allows KV positions beyond the request's pages")
        for h in range(Hq):
            hk = h // g
            oo, ll = attention_rows(q[b, h][None, :], kb[hk], vb[hk], rule, np.array([0]), b, h, 1,
                                    n_pages * page, scale, score, cur, doc_ids, bias_kv_len=kv_len_table)
            o[b, h], lse[b, h] = oo[0], ll[0]
    return o, lse
