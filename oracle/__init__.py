"""CPU oracle for the NVFP4-compressed sparse MLA decode path.

TEST INFRASTRUCTURE ONLY. This package is the slow, plain, fp64 definition of
what the CUDA path computes. Only the tests, the smoke check and the CPU
baseline leg of the benchmark may import it; the product library never does,
and it shares no code, tables or helpers with the CUDA sources.

Sources (the pages this method is described on):
  * "Prime Inference: fast, reliable serving for frontier open models"
    (Prime Intellect launch post, translated page), section "Decode: NVFP4 KV
    compression", subsections "Making room for low-latency decode" (the NVFP4
    row format) and "Native NVFP4 sparse MLA decode kernel" (what the kernel
    computes, the -1 entries).
  * "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem",
    sections "Four bits per latent value: where 352 comes from" (row table),
    "A kernel that reads four bits directly", "Prefill topology: why DEP8 holds
    five times the cache" (one 512 latent + 64 rope row per token, no head
    axis) and "Decode: TP4, and the copies it keeps" (top-2,048 positions).
  * "TokenSpeed agentic inference engine" walkthrough, section 8 "MLA KV
    layout" (the cache-write call shape) and the MLA decode benchmark example
    (softmax scale 0.07216882, page size 64).

Modules:
  codec      bf16 / FP8-E4M3 / FP4-e2m1 value codecs
  pack       NVFP4 row encoding and the paged cache write
  attention  dequantisation and sparse / dense MLA decode in fp64
  fp8rows    FP8 576-byte rows (the comparison cache format), the staged
             NVFP4 -> FP8 copy, and decode over FP8 rows
  topk       top-k position selection over indexer logits
  timing     runs the oracle on query tokens of a workload over spawned worker
             processes (the benchmark's CPU baseline and reference arm); it
             adds no arithmetic of its own

Pins: every function here is checked by tests/test_oracle_*.py against facts
that do not come from this package (the pages' row arithmetic, torch's
float8_e4m3fn conversion, exact rational brute force, closed forms, torch's
scaled_dot_product_attention in fp64).
"""
from . import codec, pack, attention, fp8rows, topk  # noqa: F401
