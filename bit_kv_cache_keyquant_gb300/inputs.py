"""Seeded synthetic inputs for the quantized-KV decode path.

This module holds no arithmetic of the method (no quantization, no
attention).  It only turns (seed, tensor id, batch row, head, element
index) into fp16 activations, so that the CPU oracle and the GPU path see
identical bytes: numpy reproduces any single (batch row, head) slice on the
host, torch produces whole tensors on the device, and both give the same
fp16 values bit for bit.

Values.  Each element draws one 32-bit counter-based hash (the murmur3
finaliser applied to a stream key plus the element index) and reads three
9-bit fields b0, b1, b2 of it.  ``x = (2*(b0+b1+b2) - 1533) * 2**-9`` is an
Irwin-Hall(3) variate: mean 0, variance 1.0000 (sum of three discrete
uniforms on 0..511), support [-2.994, 2.994], and exactly representable in
fp16 (|2S-1533| <= 1533 < 2048).  It stands in for the N(0, 1) activations
the pages' synthetic workloads use.  Per-channel multipliers (the outlier key
channels, the log-uniform per-channel sigma of the mixed-key workload) are
applied as one fp32 multiply followed by IEEE round-to-nearest to fp16, which
numpy and torch (CPU or CUDA) both perform exactly.

The five workloads (head_dim 128 throughout):

1. tiny K2V2:   B=1,  Hq=Hkv=4,  L=512,    4 seeded key channels x20
2. Llama-2-7B:  B=32, Hq=Hkv=32, L=4096
3. Llama-3-8B:  B=64, Hq=32, Hkv=8, L=32768, 1 seeded key channel / kv head x15
4. Qwen3-8B mixed key: B=16, Hq=32, Hkv=8, L=131072,
                sigma_c = 0.5 * 16**u, u ~ U[0,1) per (kv head, channel)
5. INT8 dither: B=8, Hq=64, Hkv=8, L_b ~ U{16384..65536}
"""
from __future__ import annotations

import dataclasses

import numpy as np

MASK32 = 0xFFFFFFFF
_C1 = 0x85EBCA6B
_C2 = 0xC2B2AE35
_GOLD = 0x9E3779B1

# tensor ids of the hash streams
T_K, T_V, T_Q, T_SCALE, T_LEN, T_REQ, T_OUTLIER, T_SLOT = 1, 2, 3, 4, 5, 6, 7, 8


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic decode workload."""
    index: int
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    seq_len: int                 # fixed length, or the upper bound when ragged
    variant: str                 # "kivi", "kitty", "int8", "int8t" (token-granular slot pool)
    head_dim: int = 128
    outlier_channels: int = 0    # per kv head, seeded
    outlier_gain: float = 1.0
    channel_sigma: bool = False  # per-(kv head, channel) sigma, log-uniform [0.5, 8]
    min_seq_len: int = 0         # >0: lengths ~ U{min..seq_len}
    fixed_outliers: bool = False  # same outlier channels for every kv head
    bits_k: int = 2              # KIVI code widths
    bits_v: int = 2
    paged: bool = False          # KIVI: pages of 128 tokens from a shared pool through a page table
    score_mode: int = 0          # Kitty boost selection: 0 = Eq. 2 sum of |x|, 1 = variance over the page

    @property
    def seed(self) -> int:
        return 0x5EED0000 + self.index


WORKLOADS = {
    1: Workload(1, "tiny K2V2 B1 H4 L512", 1, 4, 4, 512, "kivi",
                outlier_channels=4, outlier_gain=20.0, fixed_outliers=True),
    2: Workload(2, "Llama-2-7B-shaped MHA B32 H32 L4096", 32, 32, 32, 4096, "kivi"),
    3: Workload(3, "Llama-3-8B-shaped GQA B64 32q/8kv L32768", 64, 32, 8, 32768,
                "kivi", outlier_channels=1, outlier_gain=15.0),
    4: Workload(4, "Qwen3-8B-shaped mixed key B16 32q/8kv L131072", 16, 32, 8,
                131072, "kitty", channel_sigma=True),
    5: Workload(5, "INT8 dither B8 64q/8kv L~U[16384,65536]", 8, 64, 8, 65536,
                "int8", min_seq_len=16384),
    6: Workload(6, "INT8 token-granular slot pool B8 64q/8kv L~U[16384,65536]", 8, 64, 8, 65536,
                "int8t", min_seq_len=16384),
    7: Workload(7, "KIVI-4 Llama-2-7B-shaped MHA B32 H32 L4096", 32, 32, 32, 4096, "kivi", bits_k=4, bits_v=4),
    8: Workload(8, "paged KIVI Llama-2-7B-shaped MHA B32 H32 L4096", 32, 32, 32, 4096, "kivi", paged=True),
    9: Workload(9, "KIVI-4 Llama-3-8B-shaped GQA B64 32q/8kv L32768", 64, 32, 8, 32768, "kivi",
                outlier_channels=1, outlier_gain=15.0, bits_k=4, bits_v=4),
    10: Workload(10, "Llama-3-70B-shaped GQA B64 64q/8kv L32768", 64, 64, 8, 32768, "kivi",
                 outlier_channels=1, outlier_gain=15.0),
}


# ----------------------------------------------------------------------------
# counter-based hash (numpy: uint32 lanes, wrapping products)
# ----------------------------------------------------------------------------
def _fmix32_np(h):
    """murmur3 finaliser on uint32 arrays (products wrap modulo 2**32)."""
    h = h.astype(np.uint32, copy=True)
    h ^= h >> np.uint32(16)
    h *= np.uint32(_C1)
    h ^= h >> np.uint32(13)
    h *= np.uint32(_C2)
    h ^= h >> np.uint32(16)
    return h


def _fmix32_int(h: int) -> int:
    h &= MASK32
    h ^= h >> 16
    h = (h * _C1) & MASK32
    h ^= h >> 13
    h = (h * _C2) & MASK32
    h ^= h >> 16
    return h


def stream_key(seed: int, tensor: int, b: int, h: int) -> int:
    """32-bit key of the hash stream for one (tensor, batch row, head)."""
    k = _fmix32_int(seed ^ 0xA5A5A5A5)
    k = _fmix32_int(k ^ (tensor * 0x01000193))
    k = _fmix32_int(k ^ (b * 0x00010001 + 0x1234567))
    k = _fmix32_int(k ^ (h * 0x0000A3B1 + 0x89ABCDE))
    return k


def hash_np(key: int, index: np.ndarray) -> np.ndarray:
    """32-bit hash of (key, index) for an index array (index < 2**32), as uint64 values."""
    idx = np.asarray(index).astype(np.uint32)
    h = idx * np.uint32(_GOLD) + np.uint32(key)
    return _fmix32_np(h).astype(np.uint64)


def irwin_hall_np(hv: np.ndarray) -> np.ndarray:
    """fp32 values (2*(b0+b1+b2) - 1533) * 2**-9 from 32-bit hashes."""
    m = np.uint64(0x1FF)
    s = (hv & m) + ((hv >> np.uint64(9)) & m) + ((hv >> np.uint64(18)) & m)
    k = s.astype(np.int64) * 2 - 1533
    return k.astype(np.float32) * np.float32(2.0 ** -9)


# ----------------------------------------------------------------------------
# per-workload metadata (host, tiny)
# ----------------------------------------------------------------------------
def seq_lens(w: Workload) -> np.ndarray:
    """int32 [B] lengths (tokens in the cache including the current one)."""
    if w.min_seq_len <= 0:
        return np.full(w.batch, w.seq_len, dtype=np.int32)
    key = stream_key(w.seed, T_LEN, 0, 0)
    hv = hash_np(key, np.arange(w.batch, dtype=np.uint64))
    span = w.seq_len - w.min_seq_len + 1
    return (w.min_seq_len + (hv % np.uint64(span)).astype(np.int64)).astype(np.int32)


def request_ids(w: Workload) -> np.ndarray:
    """int32 [B] request ids (distinct, seeded)."""
    key = stream_key(w.seed, T_REQ, 0, 0)
    hv = hash_np(key, np.arange(w.batch, dtype=np.uint64))
    ids = (hv & np.uint64(0x7FFFFF00)).astype(np.int64) + np.arange(w.batch)
    return ids.astype(np.int32)


def page_permutation(w: Workload, n_pages: int) -> np.ndarray:
    """Seeded permutation of a slot pool's pages: the order in which a long-running
    allocator hands pages out, so a request's tokens land on scattered pages."""
    hv = hash_np(stream_key(w.seed, T_SLOT, 0, 0), np.arange(n_pages, dtype=np.uint64))
    return np.argsort(hv, kind="stable")


def key_channel_gain(w: Workload) -> np.ndarray:
    """fp32 [Hkv][D] multiplier applied to keys (outliers or per-channel sigma)."""
    g = np.ones((w.n_kv_heads, w.head_dim), dtype=np.float32)
    if w.outlier_channels > 0:
        for h in range(w.n_kv_heads):
            key = stream_key(w.seed, T_OUTLIER, 0, 0 if w.fixed_outliers else h)
            hv = hash_np(key, np.arange(4 * w.head_dim, dtype=np.uint64))
            chosen = []
            for v in hv.tolist():
                c = int(v % w.head_dim)
                if c not in chosen:
                    chosen.append(c)
                if len(chosen) == w.outlier_channels:
                    break
            g[h, chosen] = np.float32(w.outlier_gain)
    if w.channel_sigma:
        for h in range(w.n_kv_heads):
            key = stream_key(w.seed, T_SCALE, 0, h)
            hv = hash_np(key, np.arange(w.head_dim, dtype=np.uint64))
            u = (hv >> np.uint64(8)).astype(np.float64) * 2.0 ** -24
            g[h] = (0.5 * 16.0 ** u).astype(np.float32)
    return g


def value_channel_gain(w: Workload) -> np.ndarray:
    """fp32 [Hkv][D] multiplier applied to values (per-channel sigma only)."""
    if w.channel_sigma:
        return key_channel_gain(dataclasses.replace(w, outlier_channels=0))
    return np.ones((w.n_kv_heads, w.head_dim), dtype=np.float32)


# ----------------------------------------------------------------------------
# host generation of single slices (numpy)
# ----------------------------------------------------------------------------
def gen_slice_np(seed: int, tensor: int, b: int, h: int, n_rows: int, d: int,
                 row0: int = 0, gain: np.ndarray | None = None) -> np.ndarray:
    """fp16 [n_rows][d] rows row0.. of one (tensor, b, h) stream."""
    key = stream_key(seed, tensor, b, h)
    idx = (np.arange(row0, row0 + n_rows, dtype=np.uint64)[:, None] * np.uint64(d)
           + np.arange(d, dtype=np.uint64)[None, :])
    x = irwin_hall_np(hash_np(key, idx))
    if gain is not None:
        x = x * gain.astype(np.float32)[None, :]
    return x.astype(np.float16)


def gen_kv_np(w: Workload, tensor: int, b: int, kvh: int, n_rows: int,
              row0: int = 0) -> np.ndarray:
    """Keys (tensor=T_K) or values (T_V) of one (batch row, kv head), fp16 [n][D]."""
    gain = key_channel_gain(w)[kvh] if tensor == T_K else value_channel_gain(w)[kvh]
    if np.all(gain == 1.0):
        gain = None
    return gen_slice_np(w.seed, tensor, b, kvh, n_rows, w.head_dim, row0, gain)


def gen_q_np(w: Workload) -> np.ndarray:
    """Queries fp16 [B][Hq][D]."""
    out = np.empty((w.batch, w.n_q_heads, w.head_dim), dtype=np.float16)
    for b in range(w.batch):
        for h in range(w.n_q_heads):
            out[b, h] = gen_slice_np(w.seed, T_Q, b, h, 1, w.head_dim)[0]
    return out


# ----------------------------------------------------------------------------
# device generation (torch), bit-identical to the numpy path
# ----------------------------------------------------------------------------
def _fmix32_torch(h):
    h = h & MASK32
    h = h ^ (h >> 16)
    h = (h * _C1) & MASK32
    h = h ^ (h >> 13)
    h = (h * _C2) & MASK32
    h = h ^ (h >> 16)
    return h


def gen_slice_torch(seed: int, tensor: int, b: int, h: int, n_rows: int, d: int,
                    device, row0: int = 0, gain=None):
    """torch fp16 [n_rows][d] on `device`; equals gen_slice_np bit for bit."""
    import torch
    key = stream_key(seed, tensor, b, h)
    rows = torch.arange(row0, row0 + n_rows, dtype=torch.int64, device=device)
    idx = rows[:, None] * d + torch.arange(d, dtype=torch.int64, device=device)[None, :]
    hv = _fmix32_torch((idx * _GOLD + key) & MASK32)
    s = (hv & 0x1FF) + ((hv >> 9) & 0x1FF) + ((hv >> 18) & 0x1FF)
    x = (s * 2 - 1533).to(torch.float32) * (2.0 ** -9)
    if gain is not None:
        x = x * torch.as_tensor(gain, dtype=torch.float32, device=device)[None, :]
    return x.to(torch.float16)


def gen_kv_torch(w: Workload, tensor: int, b: int, kvh: int, n_rows: int, device,
                 row0: int = 0):
    gain = key_channel_gain(w)[kvh] if tensor == T_K else value_channel_gain(w)[kvh]
    if np.all(gain == 1.0):
        gain = None
    return gen_slice_torch(w.seed, tensor, b, kvh, n_rows, w.head_dim, device, row0, gain)


def gen_q_torch(w: Workload, device):
    import torch
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float16, device=device)
    for b in range(w.batch):
        for h in range(w.n_q_heads):
            out[b, h] = gen_slice_torch(w.seed, T_Q, b, h, 1, w.head_dim, device)[0]
    return out
