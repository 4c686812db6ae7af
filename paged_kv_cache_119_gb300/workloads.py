"""Seeded synthetic inputs for paged decode attention.

This module builds inputs only: context lengths, block tables over a randomly
permuted block pool, NaN-filled pools with the already-cached tokens written,
queries, the step's new K/V rows with their slots, and copy-on-write pairs.  It
holds none of the attention arithmetic, and both the CUDA path and the CPU
oracle consume what it produces.

The shapes follow the workloads the PagedAttention write-ups discuss
(OPT-13B / LLaMA-13B sized heads, block_size 16, contexts up to 2048 and
beyond; shared prefixes with copy-on-write, as in Figure 8 of
"PagedAttention 完全拆解" section "内存共享"); the traces and weights behind
the pages' own measurements (ShareGPT, Alpaca) are not used -- these synthetic
tensors stand in for them.

Conventions:
  * context_lens[s] counts the current token; the pool holds tokens
    0 .. L-2 before the step and the step's reshape_and_cache writes token L-1.
  * chunk workloads (``query_len`` > 1: chunked prefill, speculative
    verification) give sequence s n_s = min(query_len, L) new tokens: the pool
    holds tokens 0 .. L-n_s-1, the step writes the last n_s, and q has one row
    per new token ([sum n_s, Hq, D], rows of sequence s at query_start[s] ..).
  * block_tables rows are padded with -1 past ceil(L/B) entries.
  * every pool slot that holds no cached token is NaN, so a kernel that reads
    outside a context produces NaN instead of a plausible number.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 119000

CONFIG_SEEDS = {"tiny": 1, "opt13b": 2, "llama13b": 3, "prefix": 4, "long16": 5, "long32": 5}


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    scale: float
    num_blocks: int
    context_lens: torch.Tensor      # int32 [S]
    block_tables: torch.Tensor      # int32 [S, W]
    q: torch.Tensor                 # [S, Hq, D]
    k_cache: torch.Tensor           # [N, Hkv, B, D]
    v_cache: torch.Tensor           # [N, Hkv, B, D]
    k_new: torch.Tensor             # [T, Hkv, D]
    v_new: torch.Tensor             # [T, Hkv, D]
    slot_mapping: torch.Tensor      # int64 [T]
    copy_pairs: np.ndarray | None = None   # int64 [P, 2] (src, dst), host
    partition_size: int = 0
    query_start: torch.Tensor | None = None   # int32 [S+1] for chunk workloads
    meta: dict = field(default_factory=dict)

    @property
    def max_context_len(self) -> int:
        return int(self.meta["max_context_len"])

    @property
    def max_query_len(self) -> int:
        return int(self.meta.get("max_query_len", 1))

    @property
    def fp8(self) -> bool:
        return self.k_cache.dtype == torch.float8_e4m3fn

    def kv_bytes(self) -> int:
        """Bytes of K and V that one decode step must read (every cached token once)."""
        esz = self.k_cache.element_size()
        return int(self.meta["total_tokens"]) * self.num_kv_heads * 2 * self.head_dim * esz


def _rng(name: str, seed: int | None) -> np.random.Generator:
    return np.random.default_rng(SEED_BASE + CONFIG_SEEDS.get(name, 0) if seed is None else seed)


def _normal(shape, std: float, dtype: torch.dtype, device, gen_seed: int) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(gen_seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _assemble(name, rng, device, *, lens, Hq, Hkv, D, B, dtype, std, pool_slack=1.1,
              tables=None, num_blocks=None, filled=None, new_tokens=None, scale=None,
              copy_pairs=None, partition_size=0, extra_meta=None, chunk=None) -> Workload:
    """Common tail: pools, q, new rows, slot mapping.

    lens        : context lengths (current token included), list[int]
    tables      : optional prebuilt list of per-sequence block-id lists
    filled      : optional {block_id: tokens_already_cached} (default: derived
                  from tables, tokens 0..L-2 of each sequence)
    new_tokens  : optional list of (seq, position) pairs whose K/V rows the step
                  writes (default: position L-1 of every sequence with L > 0)
    chunk       : optional list of per-sequence new-token counts n_s <= L_s: the
                  pool then holds tokens 0 .. L-n_s-1, the step writes the rest and
                  q gets one row per new token
    """
    S = len(lens)
    if tables is None:
        need = [math.ceil(L / B) for L in lens]
        total_blocks = sum(need)
        num_blocks = max(1, math.ceil(pool_slack * total_blocks))
        perm = rng.permutation(num_blocks)
        tables, pos = [], 0
        for n in need:
            tables.append([int(x) for x in perm[pos:pos + n]])
            pos += n
    W = max(1, max((len(t) for t in tables), default=1))
    bt = np.full((S, W), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    cached = [L - (1 if chunk is None else chunk[s]) for s, L in enumerate(lens)]
    if filled is None:
        filled = {}
        for s, L in enumerate(lens):
            for j, b in enumerate(tables[s]):
                n_old = max(0, min(B, cached[s] - j * B))
                filled[b] = max(filled.get(b, 0), n_old)
    if new_tokens is None:
        new_tokens = [(s, p) for s, L in enumerate(lens) for p in range(max(cached[s], 0), L)]
    seed0 = int(rng.integers(0, 2**31 - 1))

    count = torch.zeros(num_blocks, dtype=torch.int64)
    if filled:
        ids = torch.tensor(list(filled.keys()), dtype=torch.int64)
        count[ids] = torch.tensor(list(filled.values()), dtype=torch.int64)
    count = count.to(device)
    empty = (torch.arange(B, device=device)[None, :] >= count[:, None])   # [N, B]
    empty = empty[:, None, :, None]
    shape = (num_blocks, Hkv, B, D)
    k_cache = _normal(shape, std, dtype, device, seed0 + 1).masked_fill_(empty, float("nan"))
    v_cache = _normal(shape, std, dtype, device, seed0 + 2).masked_fill_(empty, float("nan"))
    rows = S if chunk is None else int(sum(chunk))
    q = _normal((rows, Hq, D), std, dtype, device, seed0 + 3)
    T = len(new_tokens)
    k_new = _normal((T, Hkv, D), std, dtype, device, seed0 + 4)
    v_new = _normal((T, Hkv, D), std, dtype, device, seed0 + 5)
    slots = [tables[s][p // B] * B + p % B for (s, p) in new_tokens]
    slot_mapping = torch.tensor(slots, dtype=torch.int64).to(device)
    meta = {"total_tokens": int(sum(lens)), "max_context_len": int(max(lens, default=0)),
            "std": std, "new_tokens": new_tokens, "filled_blocks": len(filled)}
    query_start = None
    if chunk is not None:
        meta["max_query_len"] = int(max(chunk, default=0))
        meta["query_tokens"] = rows
        query_start = torch.tensor(np.concatenate([[0], np.cumsum(chunk)]),
                                   dtype=torch.int32).to(device)
    meta.update(extra_meta or {})
    return Workload(
        name=name, num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
        dtype=dtype, scale=(1.0 / math.sqrt(D)) if scale is None else scale,
        num_blocks=num_blocks,
        context_lens=torch.tensor(lens, dtype=torch.int32).to(device),
        block_tables=torch.from_numpy(bt).to(device), q=q, k_cache=k_cache, v_cache=v_cache,
        k_new=k_new, v_new=v_new, slot_mapping=slot_mapping,
        copy_pairs=None if copy_pairs is None else np.asarray(copy_pairs, dtype=np.int64),
        partition_size=partition_size, meta=meta, query_start=query_start)


def to_fp8(w: Workload, headroom: float = 8.0) -> Workload:
    """The same workload over E4M3 caches.  Each kv head gets its own scale,
    headroom * std / 448 * (1 + head / Hkv), so values up to `headroom` standard
    deviations stay in range and heads differ; the cached tokens become
    e4m3(fp32(x) / scale) by PyTorch's round-to-nearest-even cast (NaN stays NaN).
    q and the step's new K/V keep the model dtype; the step's cache write
    quantises them."""
    std = float(w.meta["std"])
    heads = torch.arange(w.num_kv_heads, dtype=torch.float32)
    base = headroom * std / 448.0 * (1.0 + heads / w.num_kv_heads)
    k_scale = base.to(w.k_cache.device)
    v_scale = (base * 0.75).to(w.k_cache.device)

    def quant(pool, sc):
        return (pool.float() / sc[None, :, None, None]).to(torch.float8_e4m3fn)

    meta = dict(w.meta)
    meta["kv_dtype"] = "fp8_e4m3"
    return Workload(
        name=w.name + "_fp8", num_seqs=w.num_seqs, num_q_heads=w.num_q_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
        dtype=w.dtype, scale=w.scale, num_blocks=w.num_blocks, context_lens=w.context_lens,
        block_tables=w.block_tables, q=w.q, k_cache=quant(w.k_cache, k_scale),
        v_cache=quant(w.v_cache, v_scale), k_new=w.k_new, v_new=w.v_new,
        slot_mapping=w.slot_mapping, copy_pairs=w.copy_pairs,
        partition_size=w.partition_size, meta=dict(meta, k_scale=k_scale, v_scale=v_scale),
        query_start=w.query_start)


def tiny(device="cpu", seed=None, **kw) -> Workload:
    """4 sequences, 2 heads (MHA), head_dim 64, fp32, block_size 16, a pool of 16
    physical blocks in seeded random order; lengths {1, 15, 16, 37}; N(0,1); scale 1/8."""
    rng = _rng("tiny", seed)
    lens = kw.pop("lens", [1, 15, 16, 37])
    B = 16
    need = [math.ceil(L / B) for L in lens]
    N = kw.pop("num_blocks", 16)
    perm = rng.permutation(N)
    tables, pos = [], 0
    for n in need:
        tables.append([int(x) for x in perm[pos:pos + n]])
        pos += n
    return _assemble("tiny", rng, device, lens=lens, Hq=2, Hkv=2, D=64, B=B,
                     dtype=kw.pop("dtype", torch.float32), std=1.0, tables=tables,
                     num_blocks=N, scale=0.125, **kw)


def opt13b(device="cpu", seed=None, num_seqs=64, max_len=2048, dtype=torch.float16, **kw):
    """OPT-13B-shaped decode layer: 40 MHA heads, head_dim 128, fp16, block_size 16,
    lengths uniform in [1, max_len], pool = total blocks + 10%, N(0,1)."""
    rng = _rng("opt13b", seed)
    lens = [int(x) for x in rng.integers(1, max_len + 1, size=num_seqs)]
    return _assemble("opt13b", rng, device, lens=lens, Hq=40, Hkv=40, D=128, B=16,
                     dtype=dtype, std=1.0, **kw)


def llama13b(device="cpu", seed=None, num_seqs=256, dtype=torch.bfloat16, query_len=1,
             name="llama13b", **kw):
    """LLaMA-13B-shaped batched decode: 40 MHA heads, head_dim 128, bf16, block_size 16,
    lengths lognormal (median 400, sigma 0.8) rounded and clipped to [16, 2048],
    N(0, 0.5) values, one new token per sequence (``query_len`` > 1: that many new
    tokens per sequence, attended causally, as in speculative verification)."""
    rng = _rng("llama13b", seed)
    raw = rng.lognormal(mean=math.log(400.0), sigma=0.8, size=num_seqs)
    lens = [int(min(2048, max(16, round(x)))) for x in raw]
    chunk = None if query_len == 1 else [min(query_len, L) for L in lens]
    return _assemble(name, rng, device, lens=lens, Hq=40, Hkv=40, D=128, B=16,
                     dtype=dtype, std=0.5, chunk=chunk, **kw)


def prefix(device="cpu", seed=None, num_groups=16, group_size=8, prefix_blocks=64,
           max_suffix=256, dtype=torch.bfloat16, **kw):
    """Shared-prefix / parallel-sampling decode: 32 query / 8 kv heads, head_dim 128,
    bf16, block_size 16.  Each group of ``group_size`` sequences shares
    ``prefix_blocks`` full blocks plus one partially filled tail block (f tokens,
    f in [1, 15]).  Before decode, all but the last sequence of a group take a
    copy-on-write copy of the tail block (the pairs returned in ``copy_pairs``);
    the last keeps the original.  Each sequence then appends a unique suffix of
    1..max_suffix tokens, filling its tail block first: the step's reshape_and_cache
    writes every suffix token.  L = 16 * prefix_blocks + f + suffix."""
    rng = _rng("prefix", seed)
    B = 16
    Hq, Hkv, D = 32, 8, 128
    S = num_groups * group_size
    # logical allocation order first, physical ids from a permutation afterwards
    f = [int(x) for x in rng.integers(1, B, size=num_groups)]
    u = [int(x) for x in rng.integers(1, max_suffix + 1, size=S)]
    n_logical = 0

    def new_block():
        nonlocal n_logical
        n_logical += 1
        return n_logical - 1

    tables, lens, filled_logical, pairs_logical, new_tokens = [], [], {}, [], []
    for g in range(num_groups):
        shared = [new_block() for _ in range(prefix_blocks)]
        tail = new_block()
        for b in shared:
            filled_logical[b] = B
        filled_logical[tail] = f[g]
        for i in range(group_size):
            s = g * group_size + i
            if i < group_size - 1:
                mine = new_block()
                filled_logical.setdefault(mine, 0)
                pairs_logical.append((tail, mine))
            else:
                mine = tail
            L = prefix_blocks * B + f[g] + u[s]
            need = math.ceil(L / B)
            extra = [new_block() for _ in range(need - prefix_blocks - 1)]
            for b in extra:
                filled_logical.setdefault(b, 0)
            tables.append(shared + [mine] + extra)
            lens.append(L)
            start = prefix_blocks * B + f[g]
            new_tokens.extend((s, p) for p in range(start, L))
    N = math.ceil(1.1 * n_logical)
    perm = rng.permutation(N)
    tables = [[int(perm[b]) for b in t] for t in tables]
    filled = {int(perm[b]): n for b, n in filled_logical.items()}
    pairs = [(int(perm[a]), int(perm[b])) for a, b in pairs_logical]
    return _assemble("prefix", rng, device, lens=lens, Hq=Hq, Hkv=Hkv, D=D, B=B, dtype=dtype,
                     std=1.0, tables=tables, num_blocks=N, filled=filled,
                     new_tokens=new_tokens, copy_pairs=pairs,
                     extra_meta={"tail_fill": f, "suffix": u,
                                 "unique_tokens": sum(16 * prefix_blocks + fi for fi in f)
                                 + sum(u)}, **kw)


def long_context(device="cpu", seed=None, block_size=16, num_seqs=8, context=32768,
                 dtype=torch.bfloat16, partition_size=512, query_len=1, name=None, **kw):
    """Long-context split-context decode: 64 query / 8 kv heads, head_dim 128, bf16,
    ``num_seqs`` sequences of ``context`` tokens, block_size 16 or 32, randomly
    permuted pool, N(0,1), split into ``partition_size``-token partitions.
    ``query_len`` > 1: the last ``query_len`` tokens of each context are new and
    attended causally (a chunked-prefill step)."""
    base = "long16" if block_size == 16 else "long32"
    rng = _rng(base, seed)
    lens = [int(context)] * num_seqs
    chunk = None if query_len == 1 else [min(query_len, L) for L in lens]
    return _assemble(name or base, rng, device, lens=lens, Hq=64, Hkv=8, D=128, B=block_size,
                     dtype=dtype, std=1.0, partition_size=partition_size, chunk=chunk, **kw)


CONFIGS = {
    "tiny": tiny,
    "opt13b": opt13b,
    "llama13b": llama13b,
    "prefix": prefix,
    "long16": lambda device="cpu", seed=None, **kw: long_context(device, seed, 16, **kw),
    "long32": lambda device="cpu", seed=None, **kw: long_context(device, seed, 32, **kw),
    # multi-token queries: speculative verification of 4 tokens per sequence on the
    # LLaMA-13B batch, and a 512-token chunked-prefill step on the long contexts
    "llama13b_verify4": lambda device="cpu", seed=None, **kw: llama13b(
        device, seed, **{"query_len": 4, "name": "llama13b_verify4", **kw}),
    "long16_chunk512": lambda device="cpu", seed=None, **kw: long_context(
        device, seed, 16, **{"query_len": 512, "name": "long16_chunk512", "partition_size": 0,
                             **kw}),
}


def make(name: str, device="cpu", seed=None, **overrides) -> Workload:
    """Build the named workload; keyword overrides shrink it (e.g. num_seqs=8)."""
    return CONFIGS[name](device=device, seed=seed, **overrides)
