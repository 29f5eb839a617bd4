// api.cu -- the extern "C" boundary of libspectree (declared in spec_tree.h):
// argument validation, workspace sizing and the kernel launches.
#include <stdint.h>

#include "checks.h"
#include "common.cuh"
#include "kernels.h"

namespace {

using spec::WsLayout;
using spec::al16;
using spec::check_cfg;
using spec::check_tree;

int cuda_rc(cudaError_t e) {
    if (e == cudaSuccess) return ST_OK;
    if (e == cudaErrorInvalidConfiguration) return ST_EUNSUPPORTED;
    return ST_ECUDA;
}

}  // namespace

extern "C" {

int spec_abi_version(void) { return SPEC_TREE_ABI_VERSION; }

const char* spec_status_string(int code) {
    switch (code) {
        case ST_OK: return "ok";
        case ST_EINVAL: return "invalid argument (NULL or misaligned pointer, or shape outside the limits)";
        case ST_EUNSUPPORTED: return "unsupported dtype or shape";
        case ST_ECUDA: return "CUDA launch or copy failed";
        case ST_EOVERFLOW: return "KV cache overflow: kv_len + tau > Lmax";
        case ST_TIMEOUT: return "a bounded device-side wait gave up";
        case ST_ESCRATCH: return "shape needs more than the static scratch of the no-allocation call";
        default: return "unknown status";
    }
}

size_t spec_workspace_bytes(const spec_cfg* cfg) {
    if (check_cfg(cfg) != ST_OK) return 0;
    const int sms = spec::device_sm_count();
    if (sms < 1) return 0;
    return spec::ws_layout(*cfg, sms).total;
}

size_t spec_workspace_bytes_for_sms(const spec_cfg* cfg, int num_sms) {
    if (check_cfg(cfg) != ST_OK || num_sms < 1) return 0;
    return spec::ws_layout(*cfg, num_sms).total;
}

int spec_tree_build(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                    const int32_t* root_tok, const spec_tree* out, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(out))) return rc;
    if (!al16(lat_tok) || !al16(lat_score) || !al16(root_tok) || !al16(ws)) return ST_EINVAL;
    return cuda_rc(spec::launch_tree_build(*cfg, lat_tok, lat_score, root_tok, *out, ws,
                                           static_cast<cudaStream_t>(stream)));
}

int gdn_tree_verify(const spec_cfg* cfg, const spec_tree* tree, const float* h0, const void* q,
                    const void* k, const void* v, const float* alpha, const float* beta, void* o,
                    float* c_opt, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(tree))) return rc;
    if (!al16(h0) || !al16(q) || !al16(k) || !al16(v) || !al16(alpha) || !al16(beta) || !al16(o) ||
        !al16(ws))
        return ST_EINVAL;
    if (c_opt && !al16(c_opt)) return ST_EINVAL;
    return cuda_rc(spec::launch_gdn_tree(*cfg, *tree, h0, q, k, v, alpha, beta, o, c_opt, ws,
                                         static_cast<cudaStream_t>(stream)));
}

int attn_tree_verify(const spec_cfg* cfg, const spec_tree* tree, const void* q, const void* k_tree,
                     const void* v_tree, const void* k_cache, const void* v_cache,
                     const int32_t* kv_len, void* o, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(tree))) return rc;
    if (!al16(q) || !al16(k_tree) || !al16(v_tree) || !al16(k_cache) || !al16(v_cache) ||
        !al16(kv_len) || !al16(o) || !al16(ws))
        return ST_EINVAL;
    return cuda_rc(spec::launch_attn_tree(*cfg, *tree, q, k_tree, v_tree, k_cache, v_cache, kv_len,
                                          o, ws, static_cast<cudaStream_t>(stream)));
}

namespace {
bool temperature_ok(const spec_sampling* s) {
    return s && s->temperature > 0.0f && s->temperature <= 3.0e38f && s->reserved == 0u;
}
int accept_commit_impl(const spec_cfg* cfg, const spec_tree* tree, const void* logits,
                       const spec_sampling* smp, const spec_commit_io* io, const spec_accept* out,
                       void* ws, void* stream);
}  // namespace

int accept_and_commit(const spec_cfg* cfg, const spec_tree* tree, const void* logits,
                      const spec_commit_io* io, const spec_accept* out, void* ws, void* stream) {
    return accept_commit_impl(cfg, tree, logits, nullptr, io, out, ws, stream);
}

int accept_and_commit_sampled(const spec_cfg* cfg, const spec_tree* tree, const void* logits,
                              const spec_sampling* smp, const spec_commit_io* io,
                              const spec_accept* out, void* ws, void* stream) {
    if (!temperature_ok(smp)) return ST_EINVAL;
    return accept_commit_impl(cfg, tree, logits, smp, io, out, ws, stream);
}

}  // extern "C"

namespace {
int accept_commit_impl(const spec_cfg* cfg, const spec_tree* tree, const void* logits,
                       const spec_sampling* smp, const spec_commit_io* io, const spec_accept* out,
                       void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(tree))) return rc;
    if (!io || !out || !al16(logits) || !al16(ws)) return ST_EINVAL;
    if (!al16(io->kv_len) || !al16(io->root_tok)) return ST_EINVAL;
    if (cfg->n_gdn_layers > 0 && (!al16(io->h0) || !al16(io->gdn_k) || !al16(io->gdn_v) ||
                                  !al16(io->alpha) || !al16(io->beta)))
        return ST_EINVAL;
    if (cfg->n_attn_layers > 0 && (!al16(io->k_tree) || !al16(io->v_tree) ||
                                   !al16(io->k_cache) || !al16(io->v_cache)))
        return ST_EINVAL;
    if (!al16(out->argmax) || !al16(out->accept_len) || !al16(out->accept_nodes) ||
        !al16(out->out_tok))
        return ST_EINVAL;
    return cuda_rc(spec::launch_accept_commit(*cfg, *tree, logits, *io, *out, ws,
                                              static_cast<cudaStream_t>(stream), false,
                                              smp ? &smp->temperature : nullptr,
                                              smp ? smp->seed : 0));
}
}  // namespace

extern "C" {

int spec_tree_build_ragged(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                           const int32_t* root_tok, const int32_t* m_req, int node_budget,
                           const spec_tree* out, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(out))) return rc;
    if (!al16(lat_tok) || !al16(lat_score) || !al16(root_tok) || !al16(ws)) return ST_EINVAL;
    if (m_req && !al16(m_req)) return ST_EINVAL;
    if (node_budget >= 0 && spec::budget_select_smem(*cfg) > 200 * 1024) return ST_EUNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = spec::launch_tree_build(*cfg, lat_tok, lat_score, root_tok, *out, ws, st, false,
                                            m_req);
    if (e == cudaSuccess && node_budget >= 0)
        e = spec::launch_budget_select(*cfg, *out, node_budget, st, false);
    return cuda_rc(e);
}

int spec_tree_build_markov(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_base,
                           const float* W1, const float* W2, int R, const int32_t* root_tok,
                           const spec_tree* out, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(out))) return rc;
    if (!al16(lat_tok) || !al16(lat_base) || !al16(root_tok) || !al16(ws)) return ST_EINVAL;
    if (R < 0 || R > 1024 || (R > 0 && (!al16(W1) || !al16(W2)))) return ST_EINVAL;
    if (spec::tree_markov_smem(*cfg, R) > 200 * 1024) return ST_EUNSUPPORTED;
    return cuda_rc(spec::launch_tree_markov(*cfg, lat_tok, lat_base, W1, W2, R, root_tok, *out, ws,
                                            static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// A drafter with a Markov head: lat_score then holds the base logits.
struct MarkovHead {
    const float* W1;
    const float* W2;
    int R;
};

// The fused step; m_req / node_budget as in spec_tree_build_ragged, markov as
// in spec_tree_build_markov (NULL: the plain lattice), smp as in
// accept_and_commit_sampled (NULL: the argmax).
int verify_step(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                const int32_t* m_req, int node_budget, const MarkovHead* markov,
                const spec_sampling* smp, bool persistent, const spec_tree* tree, const spec_step_io* step, const void* logits,
                const spec_commit_io* io, const spec_accept* out, void* ws, void* stream) {
    int rc = check_cfg(cfg);
    if (rc) return rc;
    if ((rc = check_tree(tree))) return rc;
    if (!step || !io || !out) return ST_EINVAL;
    if (!al16(lat_tok) || !al16(lat_score) || !al16(logits) || !al16(ws)) return ST_EINVAL;
    if (!al16(io->kv_len) || !al16(io->root_tok)) return ST_EINVAL;
    const spec_cfg& c = *cfg;
    if (c.n_gdn_layers > 0 && (!al16(io->h0) || !al16(io->gdn_k) || !al16(io->gdn_v) ||
                               !al16(io->alpha) || !al16(io->beta) || !al16(step->gdn_q) ||
                               !al16(step->gdn_o) || (step->gdn_c && !al16(step->gdn_c))))
        return ST_EINVAL;
    if (c.n_attn_layers > 0 && (!al16(io->k_tree) || !al16(io->v_tree) || !al16(io->k_cache) ||
                                !al16(io->v_cache) || !al16(step->attn_q) || !al16(step->attn_o)))
        return ST_EINVAL;
    if (!al16(out->argmax) || !al16(out->accept_len) || !al16(out->accept_nodes) ||
        !al16(out->out_tok))
        return ST_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t esz = c.io_dtype == SPEC_IO_BF16 ? 2 : 4;
    const size_t T = (size_t)c.N + 1, B = (size_t)c.B;
    auto at = [](const void* p, size_t bytes) {
        return static_cast<const char*>(p) + bytes;
    };
    // Launch order (each kernel's wait placement relies on it; see common.cuh):
    //   tree -> attention partials (layer l, merge of l-1 between) -> merge of
    //   the last attention layer -> argmax + acceptance -> GDN layers -> commit.
    // Attention starts with the tree (its cache blocks do not need it); the
    // acceptance follows the last attention layer, which is the last reader of
    // kv_len; the merge, the logits scan and the GDN layers then overlap.
    const int na = c.n_attn_layers, ng = c.n_gdn_layers;
    auto attn_args = [&](int l, const void*& q, const void*& kt, const void*& vt, const void*& kc,
                         const void*& vc, void*& o) {
        const size_t qo = (size_t)l * B * T * c.Hq * c.D * esz;
        const size_t tr = (size_t)l * B * T * c.Hkv * c.D * esz;
        const size_t ca = (size_t)l * B * c.Lmax * c.Hkv * c.D * esz;
        q = at(step->attn_q, qo);
        kt = at(io->k_tree, tr);
        vt = at(io->v_tree, tr);
        kc = at(io->k_cache, ca);
        vc = at(io->v_cache, ca);
        o = const_cast<char*>(at(step->attn_o, qo));
    };
    if (m_req && !al16(m_req)) return ST_EINVAL;
    if (node_budget >= 0 && spec::budget_select_smem(c) > 200 * 1024) return ST_EUNSUPPORTED;
    if (markov && (markov->R < 0 || markov->R > 1024 ||
                   (markov->R > 0 && (!al16(markov->W1) || !al16(markov->W2)))))
        return ST_EINVAL;
    if (markov && spec::tree_markov_smem(c, markov->R) > 200 * 1024) return ST_EUNSUPPORTED;
    cudaError_t e = markov
        ? spec::launch_tree_markov(c, lat_tok, lat_score, markov->W1, markov->W2, markov->R,
                                   io->root_tok, *tree, ws, st, true)
        : spec::launch_tree_build(c, lat_tok, lat_score, io->root_tok, *tree, ws, st, true, m_req);
    // the shared budget trims the trees before anything reads them
    if (e == cudaSuccess && node_budget >= 0)
        e = spec::launch_budget_select(c, *tree, node_budget, st, true);
    for (int l = 0; l < na && e == cudaSuccess; ++l) {
        const void *q, *kt, *vt, *kc, *vc;
        void* o;
        if (l > 0) {
            attn_args(l - 1, q, kt, vt, kc, vc, o);
            e = spec::launch_attn_merge(c, *tree, o, ws, st, true, (l - 1) & 1, true);
            if (e != cudaSuccess) break;
        }
        attn_args(l, q, kt, vt, kc, vc, o);
        e = spec::launch_attn_partial(c, *tree, q, kt, vt, kc, vc, io->kv_len, ws, st, true, l & 1);
    }
    if (persistent) {
        // the last merge, then one cooperative launch for the argmax, the
        // acceptance, the KV append and every GDN layer's verify + commit
        if (na > 0 && e == cudaSuccess) {
            const void *q, *kt, *vt, *kc, *vc;
            void* o;
            attn_args(na - 1, q, kt, vt, kc, vc, o);
            e = spec::launch_attn_merge(c, *tree, o, ws, st, true, (na - 1) & 1, /*early=*/true);
        }
        if (e == cudaSuccess)
            e = spec::launch_verify_commit(c, *tree, *step, logits, *io, *out, ws, st, true,
                                           /*tree_wait=*/na == 0);
        return cuda_rc(e);
    }
    // The last merge comes right after the last partial (it waits for it, then
    // lets the next launch start).  The acceptance then starts its scan at once
    // and lets the GDN layers start too: nothing after it reads, before its own
    // wait, anything it or the merge writes.  The tree is then complete (the
    // merge waited for the partials, which waited for the tree), unless there is
    // no attention layer: then the GDN layers wait before they read the tree.
    // The sampled acceptance keeps one CTA per SM busy through its serial
    // draw, so it lets the GDN layers start only after its wait.
    // The commit waits first: it needs the plan and the GDN layers' last read
    // of h0.
    // With the argmax acceptance and few logits rows, the last merge and the
    // acceptance are one launch (merge CTAs, then argmax CTAs): the launch it
    // saves is a large share of a small step.  With more rows the argmax CTAs
    // run better as a launch of their own (fewer registers, more CTAs per SM
    // for the scan): measured 203 -> 213 us at 24 requests, 37.4 -> 36.4 us at
    // one.
    const bool merge_accept = na > 0 && !smp && spec::merge_accept_fits(c);
    if (na > 0 && e == cudaSuccess) {
        const void *q, *kt, *vt, *kc, *vc;
        void* o;
        attn_args(na - 1, q, kt, vt, kc, vc, o);
        e = merge_accept
            ? spec::launch_merge_accept(c, *tree, o, ws, st, true, (na - 1) & 1, logits, *io, *out)
            : spec::launch_attn_merge(c, *tree, o, ws, st, true, (na - 1) & 1, /*early=*/true);
    }
    if (e == cudaSuccess && !merge_accept)
        e = smp ? spec::launch_sample_accept(c, *tree, logits, smp->temperature, smp->seed, *io,
                                             *out, ws, st, true, /*tree_early=*/na > 0,
                                             /*trigger_first=*/false)
                : spec::launch_argmax_accept(c, *tree, logits, *io, *out, ws, st, true,
                                             /*tree_early=*/na > 0, /*trigger_first=*/true);
    for (int l = 0; l < ng && e == cudaSuccess; ++l) {
        const size_t state = (size_t)l * B * c.Hv * c.dk * c.dv;
        const size_t kq = (size_t)l * B * T * c.Hk * c.dk * esz;
        const size_t vo = (size_t)l * B * T * c.Hv * c.dv;
        const size_t gate = (size_t)l * B * T * c.Hv;
        e = spec::launch_gdn_tree(c, *tree, io->h0 + state, at(step->gdn_q, kq), at(io->gdn_k, kq),
                                  at(io->gdn_v, vo * esz), io->alpha + gate, io->beta + gate,
                                  const_cast<char*>(at(step->gdn_o, vo * esz)),
                                  step->gdn_c ? step->gdn_c + vo : nullptr, ws, st, true,
                                  /*early=*/na == 0 && !smp);
    }
    if (e == cudaSuccess) e = spec::launch_commit(c, *io, *out, ws, st, true, /*early=*/true);
    return cuda_rc(e);
}

}  // namespace

extern "C" {

int spec_step_launches_persistent(const spec_cfg* cfg) {
    if (check_cfg(cfg) != ST_OK || !spec::verify_commit_supported(*cfg)) return -1;
    return 1 + 2 * cfg->n_attn_layers + 1;  // tree, partials + merges, the fused launch
}

int spec_step_launches(const spec_cfg* cfg) {
    if (check_cfg(cfg) != ST_OK) return -1;
    const int na = cfg->n_attn_layers, ng = cfg->n_gdn_layers;
    const int commit = (na + ng) > 0 ? 1 : 0;
    // tree, partials + merges (the last merge also runs the argmax when there is
    // an attention layer and few logits rows), argmax, GDN, commit
    const bool merged = na > 0 && spec::merge_accept_fits(*cfg);
    return 1 + 2 * na + (merged ? 0 : 1) + ng + commit;
}

int spec_verify_step(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                     const spec_tree* tree, const spec_step_io* step, const void* logits,
                     const spec_commit_io* io, const spec_accept* out, void* ws, void* stream) {
    return verify_step(cfg, lat_tok, lat_score, nullptr, -1, nullptr, nullptr, false, tree, step,
                       logits, io, out, ws, stream);
}

int spec_verify_step_persistent(const spec_cfg* cfg, const int32_t* lat_tok,
                                const float* lat_score, const spec_tree* tree,
                                const spec_step_io* step, const void* logits,
                                const spec_commit_io* io, const spec_accept* out, void* ws,
                                void* stream) {
    if (check_cfg(cfg) == ST_OK && !spec::verify_commit_supported(*cfg)) return ST_EUNSUPPORTED;
    return verify_step(cfg, lat_tok, lat_score, nullptr, -1, nullptr, nullptr, true, tree, step,
                       logits, io, out, ws, stream);
}

int spec_verify_step_sampled(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                             const spec_sampling* smp, const spec_tree* tree,
                             const spec_step_io* step, const void* logits,
                             const spec_commit_io* io, const spec_accept* out, void* ws,
                             void* stream) {
    if (!temperature_ok(smp)) return ST_EINVAL;
    return verify_step(cfg, lat_tok, lat_score, nullptr, -1, nullptr, smp, false, tree, step,
                       logits, io, out, ws, stream);
}

int spec_verify_step_markov(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_base,
                            const float* W1, const float* W2, int R, const spec_tree* tree,
                            const spec_step_io* step, const void* logits, const spec_commit_io* io,
                            const spec_accept* out, void* ws, void* stream) {
    const MarkovHead head{W1, W2, R};
    return verify_step(cfg, lat_tok, lat_base, nullptr, -1, &head, nullptr, false, tree, step,
                       logits, io, out, ws, stream);
}

int spec_verify_step_ragged(const spec_cfg* cfg, const int32_t* lat_tok, const float* lat_score,
                            const int32_t* m_req, int node_budget, const spec_tree* tree,
                            const spec_step_io* step, const void* logits, const spec_commit_io* io,
                            const spec_accept* out, void* ws, void* stream) {
    return verify_step(cfg, lat_tok, lat_score, m_req, node_budget, nullptr, nullptr, false, tree,
                       step, logits, io, out, ws, stream);
}

int spec_status_read(const void* ws, uint32_t* host_status, void* stream) {
    if (!ws || !host_status) return ST_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return ST_ECUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? ST_OK : ST_ECUDA;
}

int spec_status_clear(void* ws, void* stream) {
    if (!ws) return ST_EINVAL;
    return cudaMemsetAsync(ws, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ST_OK
               : ST_ECUDA;
}

}  // extern "C"
