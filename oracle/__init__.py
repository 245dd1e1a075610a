"""Plain fp64 CPU oracle for the streaming block-causal hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import or run it.  It shares no code, table or helper
with the CUDA library in ``streaming_block_causal_flash_b300/``; the two meet
only through the seeded input generators, which hold none of the method's
arithmetic.

Sources (web pages about Wan-Streamer; cited by title and section):

* "全双工语音模型精读⑫：Wan-Streamer——当全双工长出一张脸" (alwayszhang.cn),
  sections 3.1 (autoregressive factorisation), 3.2 (flow-matching interpolant
  and velocity), 3.3 (all-causal stack, 160 ms units) and 四、推理 (the
  performer appends each received KV slice to its full-history cache, then
  runs the flow solver).
* Wan Streamer real-time AV explainer (xiaohu-jiedu.pages.dev), section
  "怎么做到边听边说、随时能打断" (block-causal visibility: tokens of a block see
  each other in both directions, see every earlier block, never a later one).
* "阿里通义万相发布亚秒级同步AI视频通话基础模型" (youleyou.com), sections 3.1
  (block-causal attention over the interleaved causal sequence) and 3.3
  (performer runs only the flow-matching solver over the shared KV cache).

Functions and what pins each (tests/test_oracle_pins.py):

* ``block_causal.row_limit`` / ``visibility_mask`` -- golden block-visibility
  fixture from the explainer's four-block example; two independent
  formulations cross-checked; causal and full special cases.
* ``block_causal.attention_rows`` / ``block_causal_attention`` -- brute force
  with an explicit N x N mask; one block == full attention (torch SDPA in
  fp64); unit blocks == causal attention (torch SDPA is_causal); Q = 0 gives
  the mean of the visible V rows; constant V gives that row; LSE equals
  scipy logsumexp of the visible logits; streaming invariant.
* ``kv_cache.kv_append`` -- appending the slices of a known timeline one unit
  at a time rebuilds the timeline; bytes outside the written range unchanged.
* ``flow_matching`` -- closed form: one Euler step from tau=1 with the exact
  velocity recovers z_0; uniform k-step solve also recovers z_0; one step of
  any size moves along the straight interpolant exactly.  Guided step: w = 0
  and w = 1 give the unconditional and conditional steps exactly; with both
  velocities equal to the exact one, any w recovers z_0; the guided velocity
  is affine in w (two-point extrapolation).

No function here is "parity unpinned".
"""
