"""CPU oracle for the DFlash draft-and-verify cycle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import or run anything in this
package.  The product path (``block_speculative_decoding_gb300``) never imports
it and has no CPU fallback.

The oracle is plain numpy in float64.  It shares no code with the CUDA path:
no kernels, headers, helpers or table generators.  Each function cites the
passage of the DFlash pages it follows (page title, section, formula).

Pins (what ties each function to something other than itself) live in
``tests/test_oracle_*.py``.  Every public function is pinned; none is
"parity unpinned".
"""

from .dflash_oracle import (  # noqa: F401
    round_to_bf16,
    philox4,
    philox4x32_10,
    verify_uniforms,
    rms_norm,
    rope_inv_freq,
    rope,
    fuse_rows,
    fuse_context,
    block_attn,
    verify,
    VerifyResult,
    draft_head,
    draft_layer_qkv,
    draft_layer_tail,
    silu,
    draft_race_uniforms,
    draft_sample,
    DRAFT_TIE_EPS,
    draft_param_count,
    kv_cache_payload_bytes,
    fusion_weight_bytes,
    gather_pages,
    block_conv,
    draft_topm,
    path_score,
)
