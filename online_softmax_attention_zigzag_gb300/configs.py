"""The synthetic workloads of the ring-attention hot path, named by what they are.

Sizes follow the workloads the pages discuss: the 12-key worked example of
"Ring Attention and Ulysses shard a sequence two different ways..." (section
"Ring Attention: point-to-point rotation ..."), and long causal sequences with
grouped-query attention (8 KV heads against 64 query heads, "Interrogating
parallelism, part 5", section "Why did Llama 3 not use a ring?") cut into
zigzag chunks ("What breaks the load balance?").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    seq: int              # S
    hq: int               # query heads per batch element
    hkv: int              # key/value heads per batch element
    d: int                # head dimension
    c: int                # virtual ranks in the ring
    causal: int           # 1: token i attends to j <= i
    layout: int           # 0 contiguous (c chunks), 1 zigzag (2c chunks)
    kv_block: int         # rows per simulated ring message
    dtype: str = "bf16"   # "bf16" or "f32"
    batch: int = 1
    q_scale: float = 1.0
    outlier_frac: float = 0.0
    outlier_factor: float = 1.0
    kv_sweep: tuple = field(default_factory=tuple)
    doc_len: tuple = field(default_factory=tuple)   # (lo, hi): packed documents, all-gathered KV

    @property
    def bhq(self) -> int:
        return self.batch * self.hq

    @property
    def bhkv(self) -> int:
        return self.batch * self.hkv

    @property
    def n_chunks(self) -> int:
        return self.c * (2 if self.layout == 1 else 1)

    def flops(self) -> float:
        """Causal-adjusted attention FLOP: 4*B*Hq*d*S^2, halved when causal."""
        f = 4.0 * self.batch * self.hq * self.d * float(self.seq) ** 2
        return f * (0.5 if self.causal else 1.0)


TINY_F32 = Workload("tiny_f32_S12_d8_c3_contig_noncausal", seq=12, hq=1, hkv=1, d=8, c=3,
                    causal=0, layout=0, kv_block=4, dtype="f32")
CAUSAL_MHA_S4K = Workload("causal_mha_S4096_h8_d64_c4", seq=4096, hq=8, hkv=8, d=64, c=4,
                          causal=1, layout=1, kv_block=512)
CAUSAL_GQA_S32K = Workload("causal_gqa_S32768_h64x8_d128_c8_zigzag", seq=32768, hq=64, hkv=8,
                           d=128, c=8, causal=1, layout=1, kv_block=2048,
                           q_scale=1.0 / math.sqrt(128.0))
CAUSAL_GQA_S128K = Workload("causal_gqa_S131072_h32x8_d128_c16_zigzag", seq=131072, hq=32, hkv=8,
                            d=128, c=16, causal=1, layout=1, kv_block=4096)
NONCAUSAL_MHA_B2_S64K = Workload("noncausal_mha_B2_S65536_h16_d128_c8_contig", seq=65536, hq=16,
                                 hkv=16, d=128, c=8, causal=0, layout=0, kv_block=2048, batch=2,
                                 outlier_frac=0.01, outlier_factor=8.0,
                                 kv_sweep=(512, 1024, 2048, 4096, 8192))

# Half-length version of the 32k workload (same heads, d, c and chunking; Q 256 MiB, still
# larger than L2) for detailed counter captures, which replay each launch many times.
PROFILE_GQA_S16K = Workload("causal_gqa_S16384_h64x8_d128_c8_zigzag", seq=16384, hq=64, hkv=8,
                            d=128, c=8, causal=1, layout=1, kv_block=1024,
                            q_scale=1.0 / math.sqrt(128.0))

# All-gathered K/V with a document mask ("Interrogating parallelism, part 5", section "Why did
# Llama 3 not use a ring?"): documents of 32..8192 tokens packed into one sequence, each
# token attends causally within its own document; zigzag query chunks as in the ring.
DOCMASK_GQA_S32K = Workload("docmask_gqa_S32768_h64x8_d128_c8_zigzag", seq=32768, hq=64, hkv=8,
                            d=128, c=8, causal=1, layout=1, kv_block=2048,
                            q_scale=1.0 / math.sqrt(128.0), doc_len=(32, 8192))
# Small version for element-by-element checks: documents from 1 token up.
DOCMASK_GQA_S4K = Workload("docmask_gqa_S4096_h8x2_d128_c4_zigzag", seq=4096, hq=8, hkv=2, d=128,
                           c=4, causal=1, layout=1, kv_block=512, doc_len=(1, 2048))

WORKLOADS = {w.name: w for w in (TINY_F32, CAUSAL_MHA_S4K, CAUSAL_GQA_S32K, CAUSAL_GQA_S128K,
                                 NONCAUSAL_MHA_B2_S64K, PROFILE_GQA_S16K, DOCMASK_GQA_S32K,
                                 DOCMASK_GQA_S4K)}


def with_layout(w: Workload, layout: int) -> Workload:
    """The same workload under the other chunking (both are run for the 4096 case)."""
    from dataclasses import replace
    kv = w.kv_block
    chunk = w.seq // (w.c * (2 if layout == 1 else 1))
    if chunk % kv:
        kv = chunk
    return replace(w, layout=layout, kv_block=kv,
                   name=w.name + ("_zigzag" if layout == 1 else "_contig"))
