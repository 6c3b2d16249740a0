"""Seeded synthetic inputs for the decode workloads.

This module only draws random numbers and describes workload shapes; it
holds none of the decode arithmetic, so that the tests can feed the same
inputs to the CUDA path and to the CPU oracle without either depending on
the other.

Every draw is seeded.  Values are N(0, 1) rounded to the storage dtype, the
distribution the workloads are specified with.  Ragged lengths are uniform
integers from a CPU generator.  Cache rows that are not live are filled with a
NaN bit pattern (``POISON_BITS``) so that any read of them that reaches the
arithmetic turns the result into NaN.
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32, "int8": torch.int8}
ELEM_BYTES = {"bf16": 2, "fp16": 2, "fp32": 4, "int8": 1}
# activations (q, out, new rows) of a cache type: int8 caches take bf16 ones
ACT_DTYPE = {"bf16": "bf16", "fp16": "fp16", "fp32": "fp32", "int8": "bf16"}

# Quiet-NaN bit patterns with a recognisable payload.
POISON_BITS = {"bf16": 0x7FA5, "fp16": 0x7E5A, "fp32": 0x7FA5A5A5}
CANARY_BYTE = 0xC3


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one decode workload.

    ``prefill`` rows are already live before the first decode step (None for
    the ragged workload, whose live lengths come from ``ragged``).  ``first_append``
    is the T_new of an initial multi-row append done through the append call.
    Each of ``steps`` decode steps appends one row per sequence and attends,
    on every layer.
    """
    name: str
    n_layers: int
    batch: int
    n_heads: int
    n_kv_heads: int
    d_head: int
    max_context: int
    dtype: str
    steps: int
    prefill: int | None = None
    ragged: tuple[int, int] | None = None
    first_append: int = 0
    seed: int = 1000
    chunk: int = 0          # chunked prefill: T_new of the chunk appended after the live rows
    paged: bool = False     # cache in 16-row blocks of a pool, addressed through a block table
    d_latent: int = 0       # MLA: width of the cached latent (one row per token, no K/V heads)

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    @property
    def row_bytes(self) -> int:
        return self.d_head * ELEM_BYTES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 1 layer, MHA, 64-row prompt appended in one call, then 16 decode steps.
    "tiny_mha": Workload("tiny_mha", 1, 1, 8, 8, 32, 512, "bf16", steps=16,
                         prefill=0, first_append=64, seed=1000),
    # 12 layers, GQA 4:1, all sequences live at 512 rows, 32 decode steps.
    "small_gqa": Workload("small_gqa", 12, 8, 8, 2, 32, 1024, "bf16", steps=32,
                          prefill=512, seed=1001),
    # Llama-3-8B-shaped GQA, ragged live lengths U{1024..8192}, one step.
    "llama3_8b": Workload("llama3_8b", 32, 16, 32, 8, 128, 8192, "bf16", steps=1,
                          ragged=(1024, 8192), seed=1002),
    # Qwen2.5-1.5B-shaped GQA 6:1 at full context, fp32 and bf16 caches.
    "qwen2_5_1_5b_fp32": Workload("qwen2_5_1_5b_fp32", 28, 64, 12, 2, 128, 4096, "fp32",
                                  steps=1, prefill=4095, seed=1003),
    "qwen2_5_1_5b_bf16": Workload("qwen2_5_1_5b_bf16", 28, 64, 12, 2, 128, 4096, "bf16",
                                  steps=1, prefill=4095, seed=1013),
    # One Llama-2-70B-shaped layer (MHA 64 heads) at 32k context, B=1 and B=4.
    # The Llama-3-8B-shaped layer with an int8 cache (one fp32 scale per row).
    "llama3_8b_int8": Workload("llama3_8b_int8", 32, 16, 32, 8, 128, 8192, "int8", steps=1,
                               ragged=(1024, 8192), seed=1002),
    # The same cache paged: each sequence's live rows (and its next row) in
    # 16-row blocks placed at random in a pool of exactly those blocks.
    "llama3_8b_paged": Workload("llama3_8b_paged", 32, 16, 32, 8, 128, 8192, "bf16", steps=1,
                                ragged=(1024, 8192), seed=1002, paged=True),
    # MLA latent cache with the DeepSeek-V2 widths the pages give (d_c = 512
    # against 16 heads x 128), B=64, ragged live lengths U{1024..8192}.
    "mla_dsv2": Workload("mla_dsv2", 32, 64, 16, 1, 128, 8192, "bf16", steps=1,
                         ragged=(1024, 8192), seed=1030, d_latent=512),
    # The same latent cache read by 128 query heads (DeepSeek-V2's full head
    # count): every latent row feeds eight 16-head groups.
    "mla_dsv2_128h": Workload("mla_dsv2_128h", 32, 64, 128, 1, 128, 8192, "bf16", steps=1,
                              ragged=(1024, 8192), seed=1031, d_latent=512),
    "llama2_70b_b1": Workload("llama2_70b_b1", 1, 1, 64, 64, 128, 32768, "bf16",
                              steps=1, prefill=32767, seed=1004),
    "llama2_70b_b4": Workload("llama2_70b_b4", 1, 4, 64, 64, 128, 32768, "bf16",
                              steps=1, prefill=32767, seed=1014),
    # Multi-query attention ("10.3", section 4.1): 32 query heads share one KV
    # head of width 128; B=128 ragged U{1024..8192}, so one layer's live K/V
    # (about 300 MB) matches the Llama-3-8B-shaped GQA layer's.
    "mqa_32h": Workload("mqa_32h", 32, 128, 32, 1, 128, 8192, "bf16", steps=1,
                        ragged=(1024, 8192), seed=1040),
    # Chunked prefill on the Llama-3-8B-shaped cache: 4 sequences with live
    # prefixes U{0..4096}, a 512-token chunk each (appended, then attended).
    "llama3_8b_prefill": Workload("llama3_8b_prefill", 32, 4, 32, 8, 128, 8192, "bf16", steps=1,
                                  ragged=(0, 4096), seed=1020, chunk=512),
}


def sub_seed(seed: int, *tags) -> int:
    """A deterministic 63-bit seed derived from a base seed and tags."""
    h = hashlib.sha256(repr((seed,) + tuple(tags)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) draws rounded to ``dtype``."""
    x = torch.randn(tuple(shape), generator=generator(seed, device), device=device,
                    dtype=torch.float32)
    return x.to(DTYPES[dtype])


def ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Integers uniform on [lo, hi], inclusive, int32, on the CPU."""
    return torch.randint(lo, hi + 1, (batch,), generator=generator(seed),
                         dtype=torch.int64).to(torch.int32)


def live_lengths(w: Workload) -> torch.Tensor:
    """Live rows per sequence after the workload's one decode step (ragged),
    or after its prefill plus one step (uniform)."""
    if w.ragged is not None:
        return ragged_lengths(w.batch, w.ragged[0], w.ragged[1], sub_seed(w.seed, "len"))
    return torch.full((w.batch,), (w.prefill or 0) + w.first_append + 1, dtype=torch.int32)


BLOCK_ROWS = 16


def block_table(lengths, max_context: int, seed: int) -> tuple[np.ndarray, int]:
    """A random block table for a paged cache: sequence b gets the
    ceil(lengths[b] / 16) blocks its rows [0, lengths[b]) occupy, drawn without
    replacement from a pool of exactly the blocks all sequences need; the
    entries past those are 0 (never read).  Returns (table [B, max_context/16]
    int32, num_blocks)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    need = (lengths + BLOCK_ROWS - 1) // BLOCK_ROWS
    num_blocks = max(1, int(need.sum()))
    perm = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
    table = np.zeros((len(lengths), max_context // BLOCK_ROWS), dtype=np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, num_blocks


def poison_(t: torch.Tensor, dtype: str) -> torch.Tensor:
    """Fill a cache tensor with the NaN poison pattern, in place."""
    if dtype == "fp32":
        t.view(torch.int32).fill_(POISON_BITS[dtype])
    else:
        t.view(torch.int16).fill_(POISON_BITS[dtype] - (1 << 16) if POISON_BITS[dtype] >= 1 << 15
                                  else POISON_BITS[dtype])
    return t


def to_bits(t: torch.Tensor):
    """A CPU numpy view of a tensor's stored bits: uint16 for 16-bit types,
    float32 for fp32 (the storage forms the oracle takes)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)
