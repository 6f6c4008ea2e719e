"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws numbers.  Both the
fp64 oracle and the CUDA path consume the arrays it returns, so neither side
generates its own inputs.

Generator (portable, so x86-64 and aarch64 hosts agree bit for bit):
  * SplitMix64 counter stream: state_i = seed + (i + 1) * 0x9E3779B97F4A7C15
    (mod 2**64), output = the published SplitMix64 finaliser of state_i;
  * uniforms u = (z >> 11) * 2**-53;
  * standard normals by Box-Muller on consecutive pairs, evaluated in fp64,
    rounded to fp32, then to bf16 with round-to-nearest-even;
  * the stream of tensor `tid` under config seed `seed` is seeded with
    seed * 16 + tid.

The workloads are the ones the pages talk about: a tiny head, the
Llama-3-8B attention shape at sequence 2048 ("Fused Kernel Compiler" page,
table fusion_results), the batch 8 x 32 heads x 4096 score tensor ("Kernel
Fusion, Softmax, and Attention" page), a 32K-token context ("Optimizing LLM
Inference ..." page, FlashAttention section) and paged one-token decode over
a block table (same page, Paged Attention section).
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids within one config seed
TID_Q, TID_K, TID_V, TID_CTX, TID_PERM, TID_ROWS = 1, 2, 3, 4, 5, 6


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive SplitMix64 outputs of the stream seeded with `seed`."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniforms in [0, 1) with 53 random bits."""
    z = splitmix64(seed, n, offset)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_pairs(stream: int, first_pair: int, npairs: int) -> np.ndarray:
    """Box-Muller on SplitMix64 pairs first_pair .. first_pair+npairs-1, fp64."""
    z = splitmix64(stream, 2 * npairs, 2 * first_pair)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    pair = np.empty(2 * npairs, np.float64)
    pair[0::2] = r * np.cos(ang)
    pair[1::2] = r * np.sin(ang)
    return pair


def normal_bf16(seed: int, tid: int, shape, chunk: int = 1 << 21) -> np.ndarray:
    """i.i.d. N(0,1) values rounded to bf16, as uint16 bit patterns.

    Chunks of the counter stream are independent, so they are evaluated on
    a thread pool; the result does not depend on the chunking."""
    from concurrent.futures import ThreadPoolExecutor

    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    stream = seed * 16 + tid
    npair = (n + 1) // 2

    def work(first):
        m = min(chunk, npair - first)
        pair = _normal_pairs(stream, first, m)
        lo = 2 * first
        hi = min(n, lo + 2 * m)
        out[lo:hi] = f32_to_bf16_bits(pair[: hi - lo].astype(np.float32))

    starts = list(range(0, npair, chunk))
    if len(starts) <= 1:
        for st in starts:
            work(st)
    else:
        workers = min(len(starts), max(1, (os.cpu_count() or 1)))
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    q_mult: float = 1.0  # stability variant multiplies the bf16 Q by 8 (exact)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """4*B*Hq*Nq*Nk*d, halved under the causal mask."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def io_bytes(self) -> int:
        """Q, K, V read once, O written once (bf16), LSE written once (fp32)."""
        q = self.B * self.Hq * self.N * self.d * 2
        kv = 2 * self.B * self.Hkv * self.N * self.d * 2
        return 2 * q + kv + self.B * self.Hq * self.N * 4


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    num_seqs: int
    Hq: int
    Hkv: int
    d: int
    ctx_lo: int
    ctx_hi: int
    seed: int
    block_size: int = 16

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


PREFILL = {
    "tiny": PrefillConfig("tiny", 1, 2, 2, 128, 64, False, 1),
    "llama3_8b_causal": PrefillConfig("llama3_8b_causal", 1, 32, 8, 2048, 128, True, 2),
    "batched_noncausal": PrefillConfig("batched_noncausal", 8, 32, 32, 4096, 128, False, 3),
    "batched_causal": PrefillConfig("batched_causal", 8, 32, 32, 4096, 128, True, 3),
    "batched_stab_noncausal": PrefillConfig("batched_stab_noncausal", 8, 32, 32, 4096, 128, False, 3, 8.0),
    "batched_stab_causal": PrefillConfig("batched_stab_causal", 8, 32, 32, 4096, 128, True, 3, 8.0),
    "long_causal": PrefillConfig("long_causal", 1, 32, 8, 32768, 128, True, 4),
}

DECODE = {
    "decode_paged": DecodeConfig("decode_paged", 64, 32, 8, 128, 512, 8192, 5),
}


def prefill_inputs(cfg: PrefillConfig):
    """(q, k, v) as uint16 bf16 bits: q [B,Hq,N,d], k/v [B,Hkv,N,d]."""
    q = normal_bf16(cfg.seed, TID_Q, (cfg.B, cfg.Hq, cfg.N, cfg.d))
    if cfg.q_mult != 1.0:
        q = f32_to_bf16_bits(bf16_bits_to_f32(q) * np.float32(cfg.q_mult))
    k = normal_bf16(cfg.seed, TID_K, (cfg.B, cfg.Hkv, cfg.N, cfg.d))
    v = normal_bf16(cfg.seed, TID_V, (cfg.B, cfg.Hkv, cfg.N, cfg.d))
    return q, k, v


def prefill_inputs_shape(seed, B, Hq, Hkv, Nq, Nk, d, q_mult: float = 1.0):
    """Inputs for an arbitrary prefill shape (tests' ragged and edge cases)."""
    q = normal_bf16(seed, TID_Q, (B, Hq, Nq, d))
    if q_mult != 1.0:
        q = f32_to_bf16_bits(bf16_bits_to_f32(q) * np.float32(q_mult))
    k = normal_bf16(seed, TID_K, (B, Hkv, Nk, d))
    v = normal_bf16(seed, TID_V, (B, Hkv, Nk, d))
    return q, k, v


def ctx_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Context lengths uniform on the integers lo..hi inclusive."""
    u = uniform01(seed * 16 + TID_CTX, n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


def permutation(seed: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by the SplitMix64 stream."""
    perm = np.arange(n, dtype=np.int64)
    if n > 1:
        u = uniform01(seed * 16 + TID_PERM, n - 1)
        for idx, i in enumerate(range(n - 1, 0, -1)):
            j = int(u[idx] * (i + 1))
            perm[i], perm[j] = perm[j], perm[i]
    return perm


def paged_layout(ctx_lens: np.ndarray, block_size: int, seed: int, extra_blocks: int = 0):
    """Block table for the given context lengths.

    The pool holds sum(ceil(ctx/block_size)) (+ extra) physical blocks; a
    seeded permutation of the physical ids is handed to the logical blocks
    of all sequences in order.  Unused table entries are -1.
    Returns (block_table int32 [S, max_blocks], num_blocks)."""
    nblk = (ctx_lens.astype(np.int64) + block_size - 1) // block_size
    max_blocks = int(max(1, nblk.max() if nblk.size else 1))
    total = int(nblk.sum()) + int(extra_blocks)
    perm = permutation(seed, max(total, 1))
    table = np.full((ctx_lens.shape[0], max_blocks), -1, np.int32)
    pos = 0
    for s, nb in enumerate(nblk):
        table[s, :nb] = perm[pos:pos + nb]
        pos += int(nb)
    return table, max(total, 1)


def decode_inputs_lens(seed: int, ctx_lens, Hq: int, Hkv: int, d: int, block_size: int = 16,
                       nan_tail: bool = True, extra_blocks: int = 0):
    """Paged-decode inputs for given context lengths.

    Returns dict(q [S,Hq,d], k_cache/v_cache [num_blocks,Hkv,block_size,d]
    (uint16 bf16 bits), block_table, ctx_lens).  With nan_tail, slots past
    each sequence's last token in its last block hold NaN, so a kernel that
    reads beyond ctx_len shows it."""
    ctx_lens = np.asarray(ctx_lens, np.int32)
    S = ctx_lens.shape[0]
    table, nb = paged_layout(ctx_lens, block_size, seed, extra_blocks)
    q = normal_bf16(seed, TID_Q, (S, Hq, d))
    k = normal_bf16(seed, TID_K, (nb, Hkv, block_size, d))
    v = normal_bf16(seed, TID_V, (nb, Hkv, block_size, d))
    if nan_tail:
        nan = np.uint16(0x7FC0)
        for s in range(S):
            n = int(ctx_lens[s])
            if n % block_size and n > 0:
                phys = table[s, n // block_size]
                k[phys, :, n % block_size:, :] = nan
                v[phys, :, n % block_size:, :] = nan
    return dict(q=q, k_cache=k, v_cache=v, block_table=table, ctx_lens=ctx_lens)


def decode_inputs(cfg: DecodeConfig, nan_tail: bool = True):
    lens = ctx_lengths(cfg.seed, cfg.num_seqs, cfg.ctx_lo, cfg.ctx_hi)
    return decode_inputs_lens(cfg.seed, lens, cfg.Hq, cfg.Hkv, cfg.d, cfg.block_size, nan_tail)


def decode_kv_bytes(ctx_lens, Hkv: int, d: int) -> int:
    """Algorithmic K+V bytes one decode reads: every cached token's K and V
    row for every KV head, bf16."""
    return int(np.asarray(ctx_lens, np.int64).sum()) * Hkv * d * 2 * 2


def sample_rows(seed: int, B: int, Hq: int, Nq: int, per_head: int) -> np.ndarray:
    """per_head distinct query rows per (b, hq), seeded; int64 [B*Hq*per_head, 3]."""
    rows = []
    stream = seed * 16 + TID_ROWS
    pos = 0
    want = min(per_head, Nq)
    for b in range(B):
        for h in range(Hq):
            chosen = set()
            while len(chosen) < want:
                u = uniform01(stream, 4 * want, pos)
                pos += 4 * want
                for x in u:
                    chosen.add(int(x * Nq))
                    if len(chosen) == want:
                        break
            for i in sorted(chosen):
                rows.append((b, h, i))
    return np.asarray(rows, np.int64).reshape(-1, 3)


# ------------------------------------------------------------ add_rms_norm
@dataclass(frozen=True)
class NormConfig:
    name: str
    rows: int    # tokens
    hidden: int
    seed: int
    eps: float = 1e-6


# The shape the fusion page measures add_rms_norm on ((64, 8192) bf16), and a
# large batch of the same hidden size that streams far more than L2 holds.
NORM = {
    "rmsnorm_64x8192": NormConfig("rmsnorm_64x8192", 64, 8192, 6),
    "rmsnorm_16384x8192": NormConfig("rmsnorm_16384x8192", 16384, 8192, 7),
}


def norm_inputs_shape(seed: int, rows: int, hidden: int):
    """x, residual ~ N(0,1) bf16 [rows, hidden]; weight = 1 + 0.1 N(0,1) bf16
    [hidden] (a learned RMSNorm gain sits near one; the page gives none)."""
    x = normal_bf16(seed, 0, (rows, hidden))
    r = normal_bf16(seed, 1, (rows, hidden))
    z = bf16_bits_to_f32(normal_bf16(seed, 2, (hidden,))).astype(np.float64)
    w = f32_to_bf16_bits((1.0 + 0.1 * z).astype(np.float32))
    return x, r, w


def norm_inputs(cfg: NormConfig):
    return norm_inputs_shape(cfg.seed, cfg.rows, cfg.hidden)


# ------------------------------------------------- RoPE + paged KV-cache write
@dataclass(frozen=True)
class RopeConfig:
    name: str
    ctx_lo: int      # context length of each sequence after the write
    ctx_hi: int
    num_seqs: int
    new_tokens: int  # the last new_tokens positions of each sequence are written
    Hq: int
    Hkv: int
    d: int
    seed: int
    base: float = 500000.0  # Llama-3's rotary base


# One decode step of the paged-decode workload (one new token per sequence,
# at position ctx_len - 1) and a 16384-token prefill chunk (64 sequences x
# 256 tokens at positions 0 .. 255) of the same Llama-3-8B head layout.
ROPE = {
    "rope_decode_step": RopeConfig("rope_decode_step", 512, 8192, 64, 1, 32, 8, 128, 5),
    "rope_prefill_16k": RopeConfig("rope_prefill_16k", 256, 256, 64, 256, 32, 8, 128, 8),
}


def rope_inputs_lens(seed: int, ctx_lens, new_tokens: int, Hq: int, Hkv: int, d: int):
    """New tokens (the last new_tokens positions of each sequence, sequence by
    sequence) with q [T,Hq,d], k, v [T,Hkv,d] ~ N(0,1) bf16, their seq_ids and
    positions (int32 [T]), and the block table of the sequences' contexts.

    Returns dict(q, k, v, seq_ids, positions, block_table, num_blocks)."""
    ctx_lens = np.asarray(ctx_lens, np.int32)
    table, nb = paged_layout(ctx_lens, 16, seed)
    seq_ids, positions = [], []
    for s, n in enumerate(ctx_lens):
        first = max(0, int(n) - new_tokens)
        positions.extend(range(first, int(n)))
        seq_ids.extend([s] * (int(n) - first))
    T = len(positions)
    return dict(q=normal_bf16(seed, 0, (T, Hq, d)), k=normal_bf16(seed, 1, (T, Hkv, d)),
                v=normal_bf16(seed, 2, (T, Hkv, d)), seq_ids=np.asarray(seq_ids, np.int32),
                positions=np.asarray(positions, np.int32), block_table=table, num_blocks=nb)


def rope_inputs(cfg: RopeConfig):
    lens = ctx_lengths(cfg.seed, cfg.num_seqs, cfg.ctx_lo, cfg.ctx_hi)
    return rope_inputs_lens(cfg.seed, lens, cfg.new_tokens, cfg.Hq, cfg.Hkv, cfg.d)
