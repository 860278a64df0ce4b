"""fp64 CPU oracle for the routed MoE FFN over block-quantized experts.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package. The CUDA library never calls it, and it shares no
code with the CUDA library: no kernels, headers, helpers, tables or constants.
Its only common dependency with the GPU side is the seeded input generator in
``synth/`` (random numbers and byte placement, none of the layer's arithmetic).

What it computes (fp64 throughout; weights are the exact values decoded from
their block bytes, activations the exact bf16 values):

    out[t] = sum_j w[t, j] * W_down[e] @ ( silu(W_gate[e] @ x_t) * (W_up[e] @ x_t) ),
    e = ids[t, j],  silu(z) = z / (1 + exp(-z)),

with ids/w from a softmax top-k router and the sum taken in ascending slot j.
Sources: the routed-expert layer of "三张 RTX 3090 显卡实现 Qwen3.8-Flash-Next 80
Token 每秒的高效推理优化指南" (section 瓶颈分析: a light router picks 10 of 512
experts per token; section 优化策略三: the tiered mul_mat_id with an expert-id
range filter and the gate/up + activation fusion), and the fused SwiGLU of "一张
RTX 3090 跑 Llama 70B：三层流式缓存 + NVMe 直连" (section 4.4). The pages give no
byte layouts, router equations or combine order; the readings taken are listed
in each module's docstring.

Modules:
    formats  block decoders (Q8_0, Q4_K, Q6_K, MXFP4, IQ4_NL, IQ4_XS, IQ3_XXS, t5_g128) -> dense fp64 matrices
    router   softmax / top-k with the lower-index tie-break
    bucket   per-expert pair lists (counts, exclusive prefix sum, stable scatter)
    ffn      the layer (pair by pair, and expert by expert with bounded memory for
             full-size layers), plus an independent brute-force dense evaluation

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against hand-built blocks, closed forms, library routines (scipy softmax, numpy
lexsort) and brute force. The whole-model quality numbers of the pages
(perplexity, KLD, GSM8K) need weights and data that do not exist here: parity
unpinned for them, and nothing here claims them.
"""
from . import formats, router, bucket, ffn  # noqa: F401
