"""Float64 CPU oracle of SpargeAttn (test infrastructure only; see oracle/sparge.py)."""
from .sparge import (QBLK, KBLK, WARP_ROWS, n_blocks, default_scale, pool_sim, block_valid,
                     pooled_scores, row_softmax, count_target, topk_select, predict_mask, decisive_rows,
                     row_decisive, cut_margins, pool_key_head, predict_mask_row, attn_qblock,
                     block_sparse_attn, sparge_attn, hilbert_index_2d, hilbert_index_3d,
                     hilbert_perm_2d, hilbert_perm_3d, permute_tokens, unpermute_tokens)
