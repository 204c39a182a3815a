"""Plain, slow CPU oracle for the DeepSeek-V3-style MoE layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or call anything in this package.  The CUDA library
(``mixture_experts_layer_14_gb300``) never imports, links or calls it, and the two share
no code: the oracle is written from the definitions on the pages, in float64 numpy, with
a library matmul as the only borrowed step.

Sources (page title, section):
  * "Mixture-of-Kittens: Nhân kernel MoE nguồn mở tối ưu cho hệ thống NVL72" (aihot.vn),
    section "Chồng lấp tính toán và truyền tải trong MoE" — the layer: a router projection
    picks top-k routed experts per token with router weights; each selected expert runs a
    SwiGLU FFN (up and gate projections, SwiGLU, down projection); the shared expert and
    the routed experts are combined with the router weights.  The page's notation block and
    layer formula were lost in extraction; the plain reading used here is
        y = shared(x) + sum_{e in topk(x)} w_e * W_down_e^T (SiLU(W_gate_e^T x) * (W_up_e^T x)),
    softmax router, top-k with ties to the lower index, weights renormalised over the
    selected experts, shared expert ungated.
  * same page, section "Lập lịch" — the pull schedule: a scan over the routing tensor that
    appends each token routed to an expert, giving per-expert counts, region offsets and
    the schedule table (token index per destination row).
  * "Метод и эксперименты" (tgstat.ru) — pull dispatch: after a sort each expert reads its
    own tokens; worked example E2 <- [0,2,9,15], E5 <- [3,8], E7 <- [1,4,5,6].
  * "Mixture-of-Kittens; MoE megakernel" (news.ditty.ir), key points — bit-deterministic
    output, BF16 and MXFP8.
  * NVFP4 (oracle/nvfp4.py): the first page names it as the format of the authors' earlier
    kernels; the format definition and the recipe read from it are in that module.

Every function is pinned by tests under ``tests/`` to something other than itself
(brute force, closed forms, invariants, finite differences, the worked example, a library
conversion routine); see the docstrings for which pin covers which function.
"""

from .moe import (  # noqa: F401
    to_f64,
    router_logits,
    topk_select,
    topk_gap,
    weights_for_selection,
    route,
    dispatch,
    silu,
    expert_ffn,
    moe_forward,
    moe_forward_from_logits,
    moe_backward,
    moe_forward_mxfp8,
    moe_backward_mxfp8,
    moe_forward_nvfp4,
)
from .mxfp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_decode,
    e4m3_encode,
    mx_scale_exponent,
    mx_quantize,
    mx_dequantize,
)
from .nvfp4 import (  # noqa: F401
    E2M1_VALUES,
    e2m1_decode,
    e2m1_encode,
    nv_tensor_scale,
    nv_quantize,
    nv_dequantize,
)
