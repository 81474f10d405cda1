"""CPU fp64 oracle for the tree-verify MLA-absorb attention path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``speculative_decoding_tree_mla_gb300``) never
imports it and shares no code with it: no kernels, headers, helpers, tables
or pre/post-processing.  The only thing both sides consume is the seeded
input generator (``speculative_decoding_tree_mla_gb300.workloads``), which
holds random draws and no arithmetic of the method.
"""

from .mla_tree_attn import (  # noqa: F401
    absorb,
    ancestor_path,
    visible_positions,
    gather_cache,
    node_scores,
    softmax_rows,
    attend_latent,
    up_project,
    verify_attn_node,
    verify_attn,
    lm_head_argmax,
)
