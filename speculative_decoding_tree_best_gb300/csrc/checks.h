// checks.h -- argument checks shared by the C ABI entry points (api.cu,
// attn_noalloc.cu): every entry point returns the same ST_* code for the same
// invalid configuration or tree.
#pragma once

#include <stdint.h>

#include "spec_tree.h"

namespace spec {

inline bool al16(const void* p) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int check_cfg(const spec_cfg* c) {
    if (!c) return ST_EINVAL;
    if (c->B < 1 || c->m < 1 || c->m > SPEC_MAX_M || c->K < 1 || c->K > SPEC_MAX_K) return ST_EINVAL;
    if (c->N < 0 || c->N + 1 > SPEC_MAX_ROWS || c->V < 1 || c->Lmax < 0) return ST_EINVAL;
    if (c->Hk < 1 || c->Hv < 1 || c->Hv % c->Hk != 0) return ST_EINVAL;
    if (c->Hq < 1 || c->Hkv < 1 || c->Hq % c->Hkv != 0) return ST_EINVAL;
    if ((c->dk != 64 && c->dk != 128) || (c->dv != 64 && c->dv != 128)) return ST_EINVAL;
    if (c->D != 64 && c->D != 128) return ST_EINVAL;
    if (c->n_gdn_layers < 0 || c->n_attn_layers < 0) return ST_EINVAL;
    if (c->io_dtype != SPEC_IO_F32 && c->io_dtype != SPEC_IO_BF16) return ST_EUNSUPPORTED;
    return ST_OK;
}

inline int check_tree(const spec_tree* t) {
    if (!t) return ST_EINVAL;
    if (!al16(t->node_tok) || !al16(t->node_parent) || !al16(t->node_depth) ||
        !al16(t->node_rank) || !al16(t->node_score) || !al16(t->node_anc) || !al16(t->n_nodes))
        return ST_EINVAL;
    return ST_OK;
}

}  // namespace spec
