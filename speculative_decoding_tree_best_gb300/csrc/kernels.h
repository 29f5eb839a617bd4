// kernels.h -- launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace spec {

// pdl: launch with programmatic stream serialization (spec_verify_step only).
// m_req: lattice positions per request (nullptr: all m).
cudaError_t launch_tree_build(const spec_cfg& c, const int32_t* lat_tok, const float* lat_score,
                              const int32_t* root_tok, const spec_tree& out, void* ws,
                              cudaStream_t st, bool pdl = false, const int32_t* m_req = nullptr);
// Keep the `budget` best drafts of the batch (trees from launch_tree_build).
// cudaErrorInvalidConfiguration when the batch's scores do not fit one CTA.
cudaError_t launch_budget_select(const spec_cfg& c, const spec_tree& out, int budget,
                                 cudaStream_t st, bool pdl = false);
size_t budget_select_smem(const spec_cfg& c);

// Markov-head trees (edge scores depend on the parent's token); W1, W2 f32 [V][R].
// cudaErrorInvalidConfiguration when the edge tables exceed shared memory.
cudaError_t launch_tree_markov(const spec_cfg& c, const int32_t* lat_tok, const float* lat_base,
                               const float* W1, const float* W2, int R, const int32_t* root_tok,
                               const spec_tree& out, void* ws, cudaStream_t st, bool pdl = false);
size_t tree_markov_smem(const spec_cfg& c, int R);
size_t tree_build_smem(const spec_cfg& c);

// Returns cudaErrorInvalidConfiguration when the shape needs more shared memory
// than one CTA can have.
cudaError_t launch_gdn_tree(const spec_cfg& c, const spec_tree& t, const float* h0,
                            const void* q, const void* k, const void* v, const float* alpha,
                            const float* beta, void* o, float* c_out, void* ws, cudaStream_t st,
                            bool pdl = false, bool early = true);
size_t gdn_tree_smem(const spec_cfg& c);
// tensor-core variant (bf16 I/O, d_k = d_v = 128, T <= 32): one CTA per
// (request, v-head) state at a time; launch_gdn_tree uses it when supported
bool gdn_state_supported(const spec_cfg& c);
cudaError_t launch_gdn_state(const spec_cfg& c, const spec_tree& t, const float* h0,
                             const void* q, const void* k, const void* v, const float* alpha,
                             const float* beta, void* o, float* c_out, void* ws, cudaStream_t st,
                             bool pdl, bool early);

// The last attention layer's merge and the argmax + acceptance as one launch
// (the fused step's, with programmatic launch: the merge CTAs wait for the
// partials, the argmax CTAs scan at once).
inline bool merge_accept_fits(const spec_cfg& c) { return (long)c.B * (c.N + 1) <= 64; }
cudaError_t launch_merge_accept(const spec_cfg& c, const spec_tree& t, void* o, void* ws,
                                cudaStream_t st, bool pdl, int part_buf, const void* logits,
                                const spec_commit_io& io, const spec_accept& out);
cudaError_t launch_attn_tree(const spec_cfg& c, const spec_tree& t, const void* q,
                             const void* k_tree, const void* v_tree, const void* k_cache,
                             const void* v_cache, const int32_t* kv_len, void* o, void* ws,
                             cudaStream_t st, bool pdl = false, int part_buf = 0);

// The two halves of attn_tree_verify: split-KV partials, then the merge.
// early = false lets the merge run before its pdl_wait (only valid when the
// partials are at least two launches back).
cudaError_t launch_attn_partial(const spec_cfg& c, const spec_tree& t, const void* q,
                                const void* k_tree, const void* v_tree, const void* k_cache,
                                const void* v_cache, const int32_t* kv_len, void* ws,
                                cudaStream_t st, bool pdl, int part_buf);
cudaError_t launch_attn_merge(const spec_cfg& c, const spec_tree& t, void* o, void* ws,
                              cudaStream_t st, bool pdl, int part_buf, bool early);

bool attn_tc_supported(const spec_cfg& c);
cudaError_t launch_attn_tc(const spec_cfg& c, const spec_tree& t, const void* q,
                           const void* k_tree, const void* v_tree, const void* k_cache,
                           const void* v_cache, const int32_t* kv_len, void* ws,
                           const WsLayout& w, cudaStream_t st, bool pdl);

// accept_and_commit = argmax/accept, then the commit.  early = false lets the
// commit run before its pdl_wait (only valid when no GDN layer is the launch
// just before it).
// tree_early: the launch that wrote the tree is at least two back, so the
// kernel may read n_nodes before its programmatic wait.  trigger_first: the
// launches after it read nothing it writes before their own waits, so they may
// start at once (it still waits before the acceptance).
cudaError_t launch_argmax_accept(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl, bool tree_early,
                                 bool trigger_first = false);
// Sampled acceptance: each row's token is a draw from softmax(logits /
// temperature) (Philox4x32-10 noise keyed by seed), then the same walk.
cudaError_t launch_sample_accept(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 float temperature, uint64_t seed, const spec_commit_io& io,
                                 const spec_accept& out, void* ws, cudaStream_t st, bool pdl,
                                 bool tree_early, bool trigger_first = false);
cudaError_t launch_commit(const spec_cfg& c, const spec_commit_io& io, const spec_accept& out,
                          void* ws, cudaStream_t st, bool pdl, bool early);
// The fused, persistent verify + commit (bf16, d_k = d_v = 128, T <= 32, at
// least one GDN layer: verify_commit_supported, a host-only shape check):
// argmax + acceptance + KV append and every GDN layer's verify + commit in one
// cooperative launch; tree_wait: the tree is the previous launch.
bool verify_commit_supported(const spec_cfg& c);
cudaError_t launch_verify_commit(const spec_cfg& c, const spec_tree& t, const spec_step_io& step,
                                 const void* logits, const spec_commit_io& io,
                                 const spec_accept& out, void* ws, cudaStream_t st, bool pdl,
                                 bool tree_wait);

// temperature: nullptr for the argmax, else the sampled acceptance.
cudaError_t launch_accept_commit(const spec_cfg& c, const spec_tree& t, const void* logits,
                                 const spec_commit_io& io, const spec_accept& out, void* ws,
                                 cudaStream_t st, bool pdl = false,
                                 const float* temperature = nullptr, uint64_t seed = 0);

}  // namespace spec
