"""Seeded synthetic inputs for the FP4 indexer path.

This module only *draws inputs*: bf16 index-K rows, query heads, RoPE positions,
cache slots, page tables, per-row context lengths and head weights, plus the
model-owned bf16 RoPE cos/sin table that both the K writer and the Q packer take
as an argument ("[AMD] Enable FP4 indexer for Deepseek V4", Modifications:
deepseek_v4.py reuses the model-owned BF16 RoPE cos/sin cache).  None of the
indexer's own arithmetic (RMSNorm, RoPE rotation, Hadamard, quantisation,
logits, top-k) lives here, so the CPU oracle and the CUDA path can both consume
these inputs without sharing any of the method.

Workload shapes follow the five synthetic configurations of the indexer
benchmark: tiny decode, decode x64, draft decode x256x6, a long-context prefill
chunk and a K-store throughput case.  The pages run these on real traces and
weights (InferenceX agentic, DeepSeek-V4 checkpoints); seeded normal data of the
same shapes, length mixes and page-table structure stands in for them.
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np

HEAD_DIM = 128          # index-K / index-Q row width
N_HEADS = 64            # indexer heads
PAGE_TOKENS = 64        # compressed tokens per cache page
ROPE_DIM = 64           # rotary span: dims 0..63
ROPE_THETA = 10000.0
RMS_EPS = 1e-6
ROPE_MAX_POS = 131072   # covers every position the five workloads use


# --------------------------------------------------------------------------- bf16 inputs
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@functools.lru_cache(maxsize=4)
def rope_cos_sin_table(max_pos: int = ROPE_MAX_POS, theta: float = ROPE_THETA) -> np.ndarray:
    """Model-owned bf16 RoPE table, [max_pos, 64] uint16.

    Row p holds cos(p*f_i) in columns 0..31 and sin(p*f_i) in columns 32..63 for the
    32 frequencies f_i = theta^(-2i/64); built in float64, rounded once to bf16.
    """
    i = np.arange(ROPE_DIM // 2, dtype=np.float64)
    freq = theta ** (-2.0 * i / ROPE_DIM)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * freq[None, :]
    tab = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    out = f32_to_bf16_bits(tab)
    out.setflags(write=False)
    return out


def _normal_bf16(rng: np.random.Generator, shape, outlier_channels=None, chunk_rows=1 << 18):
    """bf16 rows ~N(0,1); the given last-dim channels are multiplied by 8."""
    shape = tuple(int(s) for s in shape)
    flat_rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    out = np.empty((flat_rows, shape[-1]), dtype=np.uint16)
    for r0 in range(0, flat_rows, chunk_rows):
        r1 = min(flat_rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, shape[-1]), dtype=np.float32)
        if outlier_channels is not None:
            x[:, outlier_channels] *= np.float32(8.0)
        out[r0:r1] = f32_to_bf16_bits(x)
    return out.reshape(shape)


# --------------------------------------------------------------------------- containers
@dataclasses.dataclass
class KStoreInputs:
    """Everything the K writer consumes (one call)."""
    k_rows: np.ndarray        # [N,128] uint16 (bf16 bits)
    positions: np.ndarray     # [N] int32 RoPE positions
    slots: np.ndarray         # [N] int32 cache slots (page*64 + j); < 0 = padding, skipped
    norm_w: np.ndarray        # [128] uint16 (bf16 RMSNorm weight)
    eps: float
    num_pages: int

    @property
    def n_rows(self) -> int:
        return int(self.k_rows.shape[0])


@dataclasses.dataclass
class IndexerInputs:
    """One decode/prefill batch: K cache contents, queries and read-side metadata."""
    name: str
    kstore: KStoreInputs      # rows that fill the K cache for every sequence
    q: np.ndarray             # [T,64,128] uint16 (bf16 bits)
    q_positions: np.ndarray   # [T] int32
    w: np.ndarray             # [T,64] float32 head weights
    page_table: np.ndarray    # [S,max_pages] int32 physical page ids (-1 = unused)
    row_seq: np.ndarray       # [T] int32 sequence of each query row
    context_lens: np.ndarray  # [T] int32 compressed tokens visible to each row
    topk: int
    seq_tokens: np.ndarray = None  # [S] int64 tokens stored per sequence (rows stored sequence by sequence)

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_pages(self) -> int:
        return self.kstore.num_pages


def _norm_weight(rng):
    return f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32))


def _head_weights(rng, t):
    # "N(0,1/8)" read as standard deviation 1/8 (= 64^-1/2, the usual per-head scale)
    return (rng.standard_normal((t, N_HEADS)) / 8.0).astype(np.float32)


def _fill_rows_for_tables(rng, seq_tokens, page_table, outliers):
    """K rows for tokens 0..L_s-1 of each sequence, stored at the slots its page table gives."""
    pos, slots = [], []
    for s, L in enumerate(seq_tokens):
        if L <= 0:
            continue
        tok = np.arange(L, dtype=np.int64)
        pos.append(tok.astype(np.int32))
        slots.append((page_table[s, tok >> 6].astype(np.int64) * PAGE_TOKENS + (tok & 63)).astype(np.int32))
    pos = np.concatenate(pos) if pos else np.zeros(0, np.int32)
    slots = np.concatenate(slots) if slots else np.zeros(0, np.int32)
    rows = _normal_bf16(rng, (pos.shape[0], HEAD_DIM), outliers)
    return rows, pos, slots


def _page_tables(rng, seq_tokens, pool_pages, permute=True):
    need = [(int(L) + PAGE_TOKENS - 1) // PAGE_TOKENS for L in seq_tokens]
    width = max(1, max(need) if need else 1)
    order = rng.permutation(pool_pages) if permute else np.arange(pool_pages)
    pt = np.full((len(seq_tokens), width), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(need):
        pt[s, :n] = order[off:off + n]
        off += n
    assert off <= pool_pages
    return pt


def _decode_q_positions(lens):
    lens = np.asarray(lens, dtype=np.int64)
    return np.where(lens > 0, 4 * lens - 1, 0).astype(np.int32)


def build_decode_batch(name, seed, seq_tokens, rows_per_seq_lens, pool_pages, topk,
                       permute_pages=True, q_outliers=True, k_outliers=True, page_table=None):
    """Generic decode/prefill batch.

    seq_tokens[s]: compressed tokens stored for sequence s.
    rows_per_seq_lens[s]: list of context lengths of the query rows of sequence s.
    """
    rng = np.random.default_rng(seed)
    ch = rng.choice(HEAD_DIM, 4, replace=False)
    norm_w = _norm_weight(rng)
    pt = page_table if page_table is not None else _page_tables(rng, seq_tokens, pool_pages, permute_pages)
    rows, pos, slots = _fill_rows_for_tables(rng, seq_tokens, pt, ch if k_outliers else None)
    lens = np.concatenate([np.asarray(r, dtype=np.int32) for r in rows_per_seq_lens])
    row_seq = np.concatenate([np.full(len(r), s, dtype=np.int32) for s, r in enumerate(rows_per_seq_lens)])
    t = lens.shape[0]
    q = _normal_bf16(rng, (t, N_HEADS, HEAD_DIM), ch if q_outliers else None)
    w = _head_weights(rng, t)
    return IndexerInputs(
        name=name,
        kstore=KStoreInputs(rows, pos, slots, norm_w, RMS_EPS, int(pool_pages)),
        q=q, q_positions=_decode_q_positions(lens), w=w, page_table=pt,
        row_seq=row_seq, context_lens=lens, topk=int(topk),
        seq_tokens=np.asarray([int(x) for x in seq_tokens], dtype=np.int64))


# --------------------------------------------------------------------------- the five workloads
def tiny_decode(seed=1000):
    """1 sequence, 1 row, L = 4,096 (64 pages, identity table), k = 512."""
    L = 4096
    b = build_decode_batch("tiny_decode_L4096_k512", seed, [L], [[L]], 64, 512,
                           permute_pages=False, q_outliers=False)
    return b


def decode_batch64(seed=1001):
    """64 sequences x 1 row, L ~ U[8192, 32768], pages from a permuted 40,960-page pool, k = 2,048."""
    rng = np.random.default_rng(seed + 7_000_000)
    L = rng.integers(8192, 32768, size=64, endpoint=True)
    return build_decode_batch("decode_b64_L8k-32k_k2048", seed, list(L), [[int(x)] for x in L],
                              40960, 2048)


def draft_batch256(seed=1002):
    """256 sequences x 6 draft rows (1,536 rows), L_r = base + r, base ~ U[1024, 17408].

    Every 8th sequence's base is moved to 61 mod 64 so its six rows cross a page
    boundary; the last 8 sequences are padding rows with context length 0.
    """
    rng = np.random.default_rng(seed + 7_000_000)
    base = rng.integers(1024, 17408, size=256, endpoint=True)
    for s in range(0, 256, 8):
        b = int(base[s]) - int(base[s]) % 64 + 61
        if b > 17408:
            b -= 64
        base[s] = b
    rows = []
    toks = []
    for s in range(256):
        if s >= 248:
            rows.append([0] * 6)
            toks.append(0)
        else:
            rows.append([int(base[s]) + r for r in range(6)])
            toks.append(int(base[s]) + 5)
    pool = sum((t + 63) // 64 for t in toks)
    return build_decode_batch("draft_b256x6_L1k-17k_k2048", seed, toks, rows, pool, 2048)


def prefill_chunk(seed=1003, rows=8192, permute_pages=False):
    """One 68k-token sequence compressed 4:1 (17,408 tokens); the last 8,192 query rows,
    causal: row t at absolute position p_t = 61,440 + t sees floor((p_t + 1) / 4) tokens."""
    Ltot = 17408
    p = 69632 - rows + np.arange(rows, dtype=np.int64)
    lens = ((p + 1) // 4).astype(np.int32)
    b = build_decode_batch("prefill_L17408_T%d_k2048" % rows, seed, [Ltot], [list(lens)], 272, 2048,
                           permute_pages=permute_pages, q_outliers=False, k_outliers=False)
    b.q_positions = p.astype(np.int32)
    return b


def kstore_65536(seed=1004):
    """65,536 rows at positions ~U[0, 131072) into the first 65,536 of a random
    permutation of the 131,072 slots of a 2,048-page cache."""
    rng = np.random.default_rng(seed)
    ch = rng.choice(HEAD_DIM, 4, replace=False)
    norm_w = _norm_weight(rng)
    n = 65536
    rows = _normal_bf16(rng, (n, HEAD_DIM), ch)
    pos = rng.integers(0, 131072, size=n).astype(np.int32)
    slots = rng.permutation(2048 * PAGE_TOKENS)[:n].astype(np.int32)
    return KStoreInputs(rows, pos, slots, norm_w, RMS_EPS, 2048)


WORKLOADS = {
    0: tiny_decode,
    1: decode_batch64,
    2: draft_batch256,
    3: prefill_chunk,
}


# --------------------------------------------------------------------------- small randomized cases
def small_batch(seed, seq_lens, rows_per_seq=1, topk=16, pool_slack=3, draft_offsets=True,
                zero_rows=(), outliers=True):
    """Small random decode batch for parity tests: ragged lengths, permuted pages.

    With rows_per_seq > 1 the rows of a sequence get lengths L - (R-1) + r (draft
    verification style); indices listed in zero_rows are padding rows (length 0).
    """
    rows = []
    toks = []
    for s, L in enumerate(seq_lens):
        r_lens = [max(0, int(L) - (rows_per_seq - 1) + r) if draft_offsets else int(L)
                  for r in range(rows_per_seq)]
        rows.append(r_lens)
        toks.append(max(r_lens) if r_lens else 0)
    flat = 0
    for s in range(len(rows)):
        for r in range(len(rows[s])):
            if flat in zero_rows:
                rows[s][r] = 0
            flat += 1
    pool = sum((t + 63) // 64 for t in toks) + pool_slack
    return build_decode_batch("small_seed%d" % seed, seed, toks, rows, max(pool, 1), topk,
                              q_outliers=outliers, k_outliers=outliers)


def small_kstore(seed, n_rows, num_pages, pad_every=0, max_pos=ROPE_MAX_POS):
    rng = np.random.default_rng(seed)
    ch = rng.choice(HEAD_DIM, 4, replace=False)
    norm_w = _norm_weight(rng)
    rows = _normal_bf16(rng, (n_rows, HEAD_DIM), ch)
    pos = rng.integers(0, max_pos, size=n_rows).astype(np.int32)
    slots = rng.permutation(num_pages * PAGE_TOKENS)[:n_rows].astype(np.int32)
    if pad_every:
        slots[::pad_every] = -1
    return KStoreInputs(rows, pos, slots, norm_w, RMS_EPS, num_pages)
