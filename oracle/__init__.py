"""FP64 CPU oracle for one Qwen-style pre-norm decoder layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The GPU library never reaches it: there is no CPU fallback.

The oracle is the plain definition of what the layer computes, written out in
numpy float64 from the BF16-rounded inputs with no intermediate rounding.  It
shares no code with the CUDA path (``transformer_decoder_layer_gb300``); the
two meet only in the seeded input generators of ``synth``.

Sources (cited by title and section throughout):

* [P1] "Qwen2.5-7B 结构拆解" (daleiyang.github.io, llm-inference-anatomy)
* [P2] "MoE 初步：参数量计算、Qwen3-30B-A3B、GQA 与 Sparse MoE" (lecture01)
* [P3] "推理系统 03：逐项算清一个真实 Qwen3 Transformer 层" (marvinlee.cn)
* [P4] "Transformer 的 Infra 视角" (inference-learning-path)
* [P5] "第七章模型容量与参数量推导" (starbuckoverflow.cn)

Parity status of each function is stated in its module; every function here is
pinned by ``tests/test_oracle_*.py`` except where a module header says
"parity unpinned".
"""

from .layer import (  # noqa: F401
    rmsnorm,
    linear,
    silu,
    sigmoid,
    rope_angles,
    apply_rope_rotate_half,
    gqa_attention,
    attention_block,
    mlp_block,
    layer_forward,
    router_topk,
    moe_block,
    moe_layer_forward,
    head_last_token,
    matmul_counted,
)
from . import counts  # noqa: F401
