"""Seeded synthetic inputs for the five paged-attention workloads.

This module only builds inputs: scheduler-side bookkeeping (which physical
blocks a sequence owns, which slot each new token goes to, its position) and
N(0, 1) activations.  It contains none of the attention step's arithmetic, so
both the CUDA path and the CPU oracle can consume exactly the same bytes.

Everything is created on the CPU with a ``torch.Generator`` seeded
``20261202 + index`` and can be copied to a device with :func:`to_device`.

Shapes come from the configurations the pages print: Qwen2-7B (hidden 3584,
28 query heads, 4 KV heads, head_dim 128, max_position_embeddings 32768,
rope_theta 1e6; "Qwen2 模型结构代码详解" section 2) and Qwen3-0.6B (16 query
heads, 8 KV heads, head_dim 128; nano-vllm Qwen3 skeleton page section 2).
Block tables and slots follow nano-vllm's per-sequence block_table and the
slot context prepare_prefill sets up (same page, section 5).

Cache slots that hold no token are filled with the bf16 pattern 0x7FC1 (a
quiet NaN), so any read or write outside the valid slots shows up.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202
SENTINEL_BF16 = 0x7FC1
BLOCK_SIZE = 16
HEAD_DIM = 128
ROPE_THETA = 1.0e6
MAX_POS = 32768

QWEN2_7B = dict(num_heads=28, num_kv_heads=4)
QWEN3_0_6B = dict(num_heads=16, num_kv_heads=8)

WORKLOAD_NAMES = [
    "tiny_qwen3_decode",      # batch 4, contexts {17, 64, 100, 255}, pool 64
    "qwen2_7b_decode_b64",    # batch 64, contexts U[128, 4096]
    "qwen2_7b_mixed_varlen",  # 4 x 512-token prefill chunks + 60 decode rows
    "qwen2_7b_long_decode",   # batch 8, every context 32768
    "qwen3_prefix_decode",    # 128 sequences sharing a 2048-token prefix
]


@dataclass
class Workload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    theta: float
    max_pos: int
    qkv: torch.Tensor            # [T, (H + 2 Hkv) D] bf16, the fused QKV rows
    positions: torch.Tensor      # [T] int32
    slot_mapping: torch.Tensor   # [T] int32
    k_cache: torch.Tensor        # [num_blocks, Hkv, BS, D] bf16
    v_cache: torch.Tensor        # [num_blocks, Hkv, BS, D] bf16
    block_tables: torch.Tensor   # [B, max_blocks_per_seq] int32
    context_lens: torch.Tensor   # [B] int32, includes the new tokens
    cu_seqlens_q: torch.Tensor   # [B + 1] int32
    q_lens: list = field(default_factory=list)
    seed: int = 0
    shared_prefix_tokens: int = 0  # tokens every table starts with in the same blocks

    # ----------------------------------------------------------- views ----
    @property
    def num_tokens(self) -> int:
        return int(self.qkv.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.num_seqs else 0

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens) if self.q_lens else 0

    @property
    def is_decode(self) -> bool:
        return all(n == 1 for n in self.q_lens)

    def q_view(self, qkv=None):
        qkv = self.qkv if qkv is None else qkv
        return qkv[:, : self.num_heads * self.head_dim]

    def k_view(self, qkv=None):
        qkv = self.qkv if qkv is None else qkv
        H, Hkv, D = self.num_heads, self.num_kv_heads, self.head_dim
        return qkv[:, H * D:(H + Hkv) * D]

    def v_view(self, qkv=None):
        qkv = self.qkv if qkv is None else qkv
        H, Hkv, D = self.num_heads, self.num_kv_heads, self.head_dim
        return qkv[:, (H + Hkv) * D:]

    def kv_bytes_read(self) -> int:
        """Bytes of K and V a decode/varlen attention pass must read:
        sum over query rows of their visible keys, counted once per
        sequence (every query of a sequence shares its keys)."""
        per_token = 2 * self.num_kv_heads * self.head_dim * self.k_cache.element_size()
        return int(self.context_lens.to(torch.int64).sum().item()) * per_token

    def unique_kv_bytes(self) -> int:
        """Bytes of distinct physical blocks referenced by the block tables."""
        per_block = (2 * self.num_kv_heads * self.block_size * self.head_dim *
                     self.k_cache.element_size())
        ids = []
        for b in range(self.num_seqs):
            nb = (int(self.context_lens[b]) + self.block_size - 1) // self.block_size
            ids.append(self.block_tables[b, :nb])
        return int(torch.unique(torch.cat(ids)).numel()) * per_block

    def causal_pairs(self) -> int:
        """(query, key) pairs of the attention, counted per query head."""
        total = 0
        for b, n in enumerate(self.q_lens):
            L = int(self.context_lens[b])
            # query i sees L - n + i + 1 keys
            total += n * (L - n) + n * (n + 1) // 2
        return total * self.num_heads


# ------------------------------------------------------------- builders ----

def _randn_bf16(gen: torch.Generator, *shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def _sentinel_cache(num_blocks, Hkv, BS, D) -> torch.Tensor:
    c = torch.full((num_blocks, Hkv, BS, D), SENTINEL_BF16, dtype=torch.int16)
    return c.view(torch.bfloat16)


def build(name_or_index, seed: int | None = None, *, scale_batch: float = 1.0,
          block_size: int = BLOCK_SIZE) -> Workload:
    """Construct one of the five workloads (by name or index 0..4).  The
    decode and mixed workloads (1-3) also come with 32- or 64-token blocks
    (same contexts and values, coarser placement)."""
    idx = name_or_index if isinstance(name_or_index, int) else WORKLOAD_NAMES.index(name_or_index)
    name = WORKLOAD_NAMES[idx]
    seed = SEED_BASE + idx if seed is None else seed
    gen = torch.Generator().manual_seed(seed)

    if idx == 0:
        shape = QWEN3_0_6B
        ctx = [17, 64, 100, 255]
        q_lens = [1] * 4
        pool = 64
        perm = torch.randperm(pool, generator=gen)
        tables, used = [], 0
        for L in ctx:
            nb = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
            tables.append(perm[used:used + nb].tolist())
            used += nb
        return _assemble(name, seed, gen, shape, ctx, q_lens, tables, pool)

    if idx == 1:
        B = max(1, int(round(64 * scale_batch)))
        ctx = torch.randint(128, 4096 + 1, (B,), generator=gen).tolist()
        return _random_placement(name, seed, gen, QWEN2_7B, ctx, [1] * B, block_size=block_size)

    if idx == 2:
        cached = torch.randint(0, 1536 + 1, (4,), generator=gen).tolist()
        dec = torch.randint(256, 2048 + 1, (60,), generator=gen).tolist()
        ctx = [c + 512 for c in cached] + dec
        q_lens = [512] * 4 + [1] * 60
        return _random_placement(name, seed, gen, QWEN2_7B, ctx, q_lens, block_size=block_size)

    if idx == 3:
        B = max(1, int(round(8 * scale_batch)))
        ctx = [MAX_POS] * B
        return _random_placement(name, seed, gen, QWEN2_7B, ctx, [1] * B, slack=0.0,
                                 block_size=block_size)

    if idx == 4:
        B = max(1, int(round(128 * scale_batch)))
        prefix_tokens = 2048
        prefix_blocks = prefix_tokens // BLOCK_SIZE
        suffix = torch.randint(64, 512 + 1, (B,), generator=gen).tolist()
        ctx = [prefix_tokens + s for s in suffix]
        unique = sum((s + BLOCK_SIZE - 1) // BLOCK_SIZE for s in suffix)
        pool = prefix_blocks + unique + max(8, unique // 10)
        perm = torch.randperm(pool, generator=gen)
        shared = perm[:prefix_blocks].tolist()
        tables, used = [], prefix_blocks
        for s in suffix:
            nb = (s + BLOCK_SIZE - 1) // BLOCK_SIZE
            tables.append(shared + perm[used:used + nb].tolist())
            used += nb
        return _assemble(name, seed, gen, QWEN3_0_6B, ctx, [1] * B, tables, pool,
                         shared_prefix_tokens=prefix_tokens)

    raise ValueError(name_or_index)


def custom(num_heads, num_kv_heads, ctx, q_lens, seed=1, pool_slack=0.1,
           shared_prefix_tokens=0, block_size=BLOCK_SIZE) -> Workload:
    """A workload with explicit context lengths and query counts, random
    block placement (used by edge-case tests); ``block_size`` tokens per
    cache block (16, 32 or 64)."""
    gen = torch.Generator().manual_seed(seed)
    shape = dict(num_heads=num_heads, num_kv_heads=num_kv_heads)
    BS = block_size
    if shared_prefix_tokens:
        # every table starts with the same blocks for the first
        # shared_prefix_tokens tokens (a multiple of the block size)
        assert shared_prefix_tokens % BS == 0
        pb = shared_prefix_tokens // BS
        own = [max(0, (L + BS - 1) // BS - pb) for L in ctx]
        pool = pb + sum(own) + max(8, int(sum(own) * pool_slack)) + 1
        perm = torch.randperm(pool, generator=gen)
        shared = perm[:pb].tolist()
        tables, used = [], pb
        for nb in own:
            tables.append(shared + perm[used:used + nb].tolist())
            used += nb
        return _assemble("custom", seed, gen, shape, list(ctx), list(q_lens), tables, pool,
                         shared_prefix_tokens=shared_prefix_tokens, block_size=BS)
    return _random_placement("custom", seed, gen, shape, list(ctx), list(q_lens),
                             slack=pool_slack, block_size=BS)


def _random_placement(name, seed, gen, shape, ctx, q_lens, slack=0.1, block_size=BLOCK_SIZE):
    need = [(L + block_size - 1) // block_size for L in ctx]
    total = sum(need)
    pool = total + int(total * slack) + 1
    perm = torch.randperm(pool, generator=gen)
    tables, used = [], 0
    for nb in need:
        tables.append(perm[used:used + nb].tolist())
        used += nb
    return _assemble(name, seed, gen, shape, ctx, q_lens, tables, pool, block_size=block_size)


def _assemble(name, seed, gen, shape, ctx, q_lens, tables, pool,
              shared_prefix_tokens=0, block_size=BLOCK_SIZE) -> Workload:
    H, Hkv = shape["num_heads"], shape["num_kv_heads"]
    D, BS = HEAD_DIM, block_size
    B = len(ctx)
    max_blocks = max(1, max(len(t) for t in tables))
    bt = torch.zeros((B, max_blocks), dtype=torch.int32)
    for b, t in enumerate(tables):
        if t:
            bt[b, : len(t)] = torch.tensor(t, dtype=torch.int32)
    k_cache = _sentinel_cache(pool, Hkv, BS, D)
    v_cache = _sentinel_cache(pool, Hkv, BS, D)

    # Already-cached tokens (positions 0 .. L - q_len - 1): N(0, 1) K and V
    # written at their slots.  Shared prefix blocks are written once.
    done_blocks = set()
    for b in range(B):
        n_cached = ctx[b] - q_lens[b]
        if n_cached <= 0:
            continue
        pos = torch.arange(n_cached)
        blk = bt[b, pos // BS].to(torch.int64)
        off = (pos % BS).to(torch.int64)
        if shared_prefix_tokens:
            keep = torch.tensor([(int(x) not in done_blocks) or (p >= shared_prefix_tokens)
                                 for x, p in zip(blk.tolist(), pos.tolist())])
            done_blocks.update(blk[: min(n_cached, shared_prefix_tokens)].tolist())
            blk, off = blk[keep], off[keep]
        n = int(blk.numel())
        if n == 0:
            continue
        k_cache[blk, :, off, :] = _randn_bf16(gen, n, Hkv, D)
        v_cache[blk, :, off, :] = _randn_bf16(gen, n, Hkv, D)

    T = sum(q_lens)
    qkv = _randn_bf16(gen, T, (H + 2 * Hkv) * D)
    positions = torch.empty(T, dtype=torch.int32)
    slots = torch.empty(T, dtype=torch.int32)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    t = 0
    for b in range(B):
        n = q_lens[b]
        for i in range(n):
            p = ctx[b] - n + i
            positions[t] = p
            slots[t] = int(bt[b, p // BS]) * BS + p % BS
            t += 1
        cu[b + 1] = t
    return Workload(name=name, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                    block_size=BS, theta=ROPE_THETA, max_pos=MAX_POS, qkv=qkv,
                    positions=positions, slot_mapping=slots, k_cache=k_cache,
                    v_cache=v_cache, block_tables=bt,
                    context_lens=torch.tensor(ctx, dtype=torch.int32),
                    cu_seqlens_q=cu, q_lens=list(q_lens), seed=seed,
                    shared_prefix_tokens=shared_prefix_tokens)


def to_device(w: Workload, device) -> Workload:
    """A copy of the workload with every tensor on ``device``."""
    kw = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
          for k, v in w.__dict__.items()}
    return Workload(**kw)


def permute_blocks(w: Workload, seed: int = 7) -> Workload:
    """The same logical cache with physical block ids relabelled by a random
    permutation pi: block_tables -> pi(block_tables), pool[pi(x)] = pool[x],
    slots follow their block."""
    gen = torch.Generator().manual_seed(seed)
    n = w.num_blocks
    pi = torch.randperm(n, generator=gen)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[pi] = w.k_cache
    v2[pi] = w.v_cache
    bt2 = pi[w.block_tables.to(torch.int64)].to(torch.int32)
    BS = w.block_size
    s = w.slot_mapping.to(torch.int64)
    s2 = torch.where(s >= 0, pi[torch.clamp(s, min=0) // BS] * BS + s % BS, s).to(torch.int32)
    kw = dict(w.__dict__)
    kw.update(k_cache=k2, v_cache=v2, block_tables=bt2, slot_mapping=s2)
    return Workload(**kw)


# FP8 caches: the per-tensor scales the workloads use (|x| / scale stays well
# inside e4m3's +-448 for N(0, 1) data).
FP8_K_SCALE = 0.0135
FP8_V_SCALE = 0.0115


def fp8_codes(cache: torch.Tensor, scale: float) -> torch.Tensor:
    """Synthetic e4m3 cache contents: the bf16 cache (cached tokens N(0, 1),
    unused slots NaN) divided by ``scale`` and converted with torch's
    float8_e4m3fn cast, as uint8 codes.  Input generation only -- which
    codes they are does not matter, both sides read the same ones."""
    x = (cache.float() / scale).clamp(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def with_fp8_cache(w: Workload, k_scale: float = FP8_K_SCALE,
                   v_scale: float = FP8_V_SCALE) -> Workload:
    """The workload with uint8 e4m3 caches in place of the bf16 ones."""
    kw = dict(w.__dict__)
    kw.update(k_cache=fp8_codes(w.k_cache, k_scale), v_cache=fp8_codes(w.v_cache, v_scale))
    return Workload(**kw)
