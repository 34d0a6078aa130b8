"""The five seeded synthetic workloads of masked attention over a BlockMask, as plain data.

A workload is shapes + a mask rule + a score rule + seeded inputs. Rules are data (lists of tuples), read
independently by the oracle and by the C-ABI marshalling; this module holds none of the method's arithmetic.

Mask rule spec: a postfix program, one tuple per op:
    ("true",) ("causal",) ("window", W) ("prefix", P) ("doc",) ("and",) ("or",)
with the meanings of FlexAttention's mask_mod examples ("FlexAttention: from rules to fused kernels",
section 1.1): causal i >= j, left window i - j < W (the window includes the current token), prefix j < P,
document equality d_b(i) == d_b(j); "and"/"or" are and_masks/or_masks. i is the GLOBAL query position
(query index + per-batch offset, "FlexAttention: compiler optimisation of custom attention", section 6).

Score rule spec: dict(alibi_slopes=[Hq] or None, rel_bias=[Hq, 2*KV_LEN-1] or None, softcap=c or 0.0).

Inputs: splitmix64 -> Box-Muller N(0,1) -> bf16 (RNE), seed 0x5EED0000 + k for workload k,
tensor ids Q=1, K=2, V=3, document lengths=4, KV lengths=5, page permutation=6.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import synth

TID_Q, TID_K, TID_V, TID_DOC, TID_KVLEN, TID_PERM, TID_DOUT = 1, 2, 3, 4, 5, 6, 7


def seed_for(k: int) -> int:
    return 0x5EED0000 + k


@dataclass
class Prefill:
    name: str
    B: int
    Hq: int
    Hkv: int
    q_len: int
    kv_len: int
    d: int
    bq: int
    bk: int
    rule: list
    score: dict
    scale: float
    seed: int
    doc_lens: Optional[np.ndarray] = None      # packed document lengths (one sequence, shared by all b)
    # filled by generate():
    q_bits: Optional[np.ndarray] = None          # uint16 [B,Hq,q_len,d]
    k_bits: Optional[np.ndarray] = None          # uint16 [B,Hkv,kv_len,d]
    v_bits: Optional[np.ndarray] = None
    doc_ids: Optional[np.ndarray] = None         # int32 [1, kv_len] (or None)
    meta: dict = field(default_factory=dict)

    def dout_bits(self) -> np.ndarray:
        """Seeded upstream gradient for the backward, bf16 bits [B,Hq,q_len,d] ~ N(0,1)."""
        return synth.normal_bf16_bits(self.seed, TID_DOUT, (self.B, self.Hq, self.q_len, self.d))

    def generate(self) -> "Prefill":
        self.q_bits = synth.normal_bf16_bits(self.seed, TID_Q, (self.B, self.Hq, self.q_len, self.d))
        self.k_bits = synth.normal_bf16_bits(self.seed, TID_K, (self.B, self.Hkv, self.kv_len, self.d))
        self.v_bits = synth.normal_bf16_bits(self.seed, TID_V, (self.B, self.Hkv, self.kv_len, self.d))
        return self


def doc_lengths(seed: int, total: int, lo: int = 256, hi: int = 4096) -> np.ndarray:
    """Draw lengths uniform on [lo, hi] until they sum to >= total; the last one is truncated."""
    lens, cur, s = [], 0, 0
    while s < total:
        v, cur = synth.uniform_ints(seed, TID_DOC, lo, hi, 1, cur)
        v = int(v[0])
        v = min(v, total - s)
        lens.append(v)
        s += v
    return np.asarray(lens, dtype=np.int64)


def doc_ids_from_lengths(lens: np.ndarray) -> np.ndarray:
    """doc(t) = k for t in [sum_{<k} len, sum_{<=k} len)."""
    return np.repeat(np.arange(len(lens), dtype=np.int32), lens.astype(np.int64))


def alibi_slopes(Hq: int) -> np.ndarray:
    """slope_h = 2^(-8(h+1)/Hq) (the ALiBi geometric sequence), fp32 values."""
    return np.asarray([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=np.float32)


def cfg1(n: int = 512) -> Prefill:
    """Tiny GQA sliding window + soft-cap: B=1, Hq=4, Hkv=2, N=512, d=64, causal & i-j<128, 20*tanh(s/20)."""
    return Prefill("cfg1_gqa_window_softcap", 1, 4, 2, n, n, 64, 64, 64,
                   [("causal",), ("window", 128), ("and",)], dict(softcap=20.0), 1.0 / 8.0, seed_for(1))


def cfg2(B: int = 4, H: int = 16, n: int = 4096) -> Prefill:
    """Plain causal: B=4, Hq=Hkv=16, N=4096, d=128, no score rule, Bq=Bk=128."""
    return Prefill("cfg2_causal", B, H, H, n, n, 128, 128, 128, [("causal",)], {}, 1.0 / math.sqrt(128),
                   seed_for(2))


def cfg3(n: int = 16384, Hq: int = 32, Hkv: int = 8) -> Prefill:
    """Packed document-causal + ALiBi: B=1, N=16384, Hq=32, Hkv=8, d=128, doc lengths U[256,4096]."""
    seed = seed_for(3)
    lens = doc_lengths(seed, n)
    w = Prefill("cfg3_doc_causal_alibi", 1, Hq, Hkv, n, n, 128, 128, 128,
                [("causal",), ("doc",), ("and",)], dict(alibi_slopes=alibi_slopes(Hq)), 1.0 / math.sqrt(128),
                seed, doc_lens=lens)
    w.doc_ids = doc_ids_from_lengths(lens).reshape(1, n)
    return w


def cfg4(n: int = 65536, H: int = 16, window: int = 1024) -> Prefill:
    """Long sliding window + soft-cap: B=1, Hq=Hkv=16, N=65536, d=128, causal & i-j<1024, 50*tanh(s/50)."""
    return Prefill(f"cfg4_window{window}_softcap_n{n}", 1, H, H, n, n, 128, 128, 128,
                   [("causal",), ("window", window), ("and",)], dict(softcap=50.0), 1.0 / math.sqrt(128),
                   seed_for(4))


@dataclass
class Decode:
    name: str
    Bz: int
    Hq: int
    Hkv: int
    d: int
    page: int
    max_pages: int
    kv_lens: np.ndarray           # int64 [Bz]
    page_table: np.ndarray        # int32 [Bz, max_pages], -1 past the request's pages
    n_pages_total: int
    rule: list
    score: dict
    scale: float
    seed: int
    fill_past_len: float = 1.0e4
    q_bits: Optional[np.ndarray] = None       # uint16 [Bz,Hq,d]
    k_bits: Optional[np.ndarray] = None       # uint16 [P_tot,Hkv,page,d]
    v_bits: Optional[np.ndarray] = None

    @property
    def kv_len(self) -> int:
        return self.max_pages * self.page

    @property
    def q_offset(self) -> np.ndarray:
        """cur_pos_b = L_b - 1: the new token's K/V already sits in the cache at slot L_b - 1."""
        return (self.kv_lens - 1).astype(np.int32)

    def generate(self) -> "Decode":
        P, H, pg, d = self.n_pages_total, self.Hkv, self.page, self.d
        self.q_bits = synth.normal_bf16_bits(self.seed, TID_Q, (self.Bz, self.Hq, d))
        self.k_bits = synth.normal_bf16_bits(self.seed, TID_K, (P, H, pg, d))
        self.v_bits = synth.normal_bf16_bits(self.seed, TID_V, (P, H, pg, d))
        fill = synth.bf16_bits_from_double(self.fill_past_len)
        for b in range(self.Bz):
            L = int(self.kv_lens[b])
            n = -(-L // pg)
            if L % pg:
                p = int(self.page_table[b, n - 1])
                self.k_bits[p, :, L % pg:, :] = fill
                self.v_bits[p, :, L % pg:, :] = fill
        return self


def cfg5(Bz: int = 64, Hq: int = 32, Hkv: int = 8, d: int = 128, page: int = 128, lo: int = 1024,
         hi: int = 32768, prefix: int = 0) -> Decode:
    """Paged decode: 64 requests x 1 token, Hq=32, Hkv=8, d=128, L_b ~ U[1024, 32768], 128-token pages
    scattered by a seeded Fisher-Yates permutation; mask kv_idx <= cur_pos (optionally OR kv_idx < prefix)."""
    seed = seed_for(5)
    lens, _ = synth.uniform_ints(seed, TID_KVLEN, lo, hi, Bz)
    max_pages = -(-hi // page)
    npages = [-(-int(L) // page) for L in lens]
    ptot = int(sum(npages))
    perm = synth.permutation(seed, TID_PERM, ptot)
    table = np.full((Bz, max_pages), -1, dtype=np.int32)
    pos = 0
    for b in range(Bz):
        table[b, :npages[b]] = perm[pos:pos + npages[b]]
        pos += npages[b]
    rule = [("causal",)] if prefix <= 0 else [("causal",), ("prefix", prefix), ("or",)]
    return Decode(f"cfg5_paged_decode{'_prefix%d' % prefix if prefix > 0 else ''}", Bz, Hq, Hkv, d, page,
                  max_pages, lens, table, ptot, rule, {}, 1.0 / math.sqrt(d), seed)


def paged_kv(bits: np.ndarray, page: int, seed: int):
    """Contiguous K or V bits [B, Hkv, N, d] -> pages [B * ceil(N / page), Hkv, page, d] at seeded shuffled
    physical ids, and the page table int32 [B, ceil(N / page)] (slots past N hold zeros)."""
    B, Hkv, N, d = bits.shape
    npg = -(-N // page)
    perm = synth.permutation(seed, TID_PERM, B * npg).astype(np.int32)
    padded = np.zeros((B, Hkv, npg * page, d), dtype=bits.dtype)
    padded[:, :, :N] = bits
    logical = padded.reshape(B, Hkv, npg, page, d).transpose(0, 2, 1, 3, 4).reshape(B * npg, Hkv, page, d)
    pages = np.empty_like(logical)
    pages[perm] = logical
    return pages, perm.reshape(B, npg)


def bf16_torch(bits: np.ndarray, device=None):
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor (a byte-for-byte view, no rounding)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t if device is None else t.to(device)
