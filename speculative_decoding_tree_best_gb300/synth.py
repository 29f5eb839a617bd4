"""Seeded synthetic inputs for the tree-verification step.

This module is the only code that the CUDA path and the CPU oracle both use:
it draws random inputs and holds none of the method's arithmetic (no tree
building, no recurrence, no attention, no acceptance).  The one data-dependent
step, planting the target's argmax, takes the tree's node depths as an input.

Workloads (shapes and value distributions of the paper digest's setting:
parallel-drafter lattices of top-16 candidates over 8 or 16 positions, a
hybrid Gated-DeltaNet / attention target, a 151936-token vocabulary):

  tiny      1 request, fp32 I/O, 4x4 lattice, N=8, 4 GDN heads of 64x64,
            4 attention heads of 64, KV 128, vocab 1024, plant p=0.8
  single    1 request, bf16 I/O, 8x16 lattice, N=24, GDN 16 qk / 32 v heads of
            128x128, attention 32 q / 8 kv heads of 128, KV 4096, vocab 151936,
            plant p=0.85
  long      1 request, 16x16 lattice, N=64, KV 16384, plant p=0.9
  batched   24 requests of 'single', KV length per request ~ U[1024, 8192]
  stack     8 requests of 'single', 48 GDN + 16 attention layers, KV 8192
  ragged    24 requests, 16x16 lattices of which request b drafts from 16, 12
            or 8 positions (cycled), a 192-node budget shared by the batch,
            N = 24 per request, KV as 'batched'
  markov    'single' with a Markov-head drafter: base logits ~ N(0, 2^2) and
            two tables W1, W2 [V][32] ~ N(0, 32^-1/2)
  sampled   'single' verified by sampling at temperature 1, planted logits at
            the row maximum + 10 (about 0.88 of the row's probability)

Value recipe: lattice scores are log-softmax over the K candidate logits
~ N(0, 2^2) of each position; candidate tokens are drawn uniformly without
replacement from the vocabulary; committed GDN state ~ N(0, 0.1^2); GDN q and k
~ N(0, 1) normalised to unit L2 norm in fp32, then rounded to the I/O type;
v ~ N(0, 1); beta = sigmoid(N(0, 1)); alpha ~ U[0.9, 1.0]; attention q, k, v
and cache ~ N(0, 1); target logits ~ N(0, 1).  For a tree node at depth d < m
the logit of the top-scoring candidate of lattice position d (0-based, i.e. the
candidate set of depth d+1) is, with probability p, set to the row maximum
plus 1.0, so that node's argmax agrees with the drafter's first choice.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import torch

__all__ = ["SpecConfig", "CONFIGS", "config", "make_lattice", "make_gdn_layer",
           "make_attn_layer", "make_kv_len", "make_logits", "plant_logits",
           "top_candidates", "row_generator", "make_step_inputs"]


@dataclasses.dataclass(frozen=True)
class SpecConfig:
    name: str
    B: int            # requests
    m: int            # lattice positions
    K: int            # candidates per position
    N: int            # draft nodes (tree rows T = N + 1)
    Hk: int           # GDN q/k heads
    Hv: int           # GDN v heads
    dk: int
    dv: int
    Hq: int           # attention query heads
    Hkv: int          # attention kv heads
    D: int            # attention head dim
    L: int            # KV length (upper end of the range when L_lo is set)
    V: int            # vocabulary
    p_plant: float
    n_gdn: int = 1
    n_attn: int = 1
    io: str = "bf16"  # "bf16" or "f32"
    L_lo: Optional[int] = None   # per-request KV length ~ U[L_lo, L] when set
    headroom: int = 64           # cache rows beyond the longest KV length
    m_cycle: Optional[tuple] = None   # draft positions per request, cycled over b
    budget: int = -1             # draft nodes shared by the batch (< 0: none)
    markov_R: int = 0            # > 0: a drafter with a Markov head of this rank
    temperature: float = 0.0     # > 0: sampled acceptance at this temperature
    sample_seed: int = 0         # the sampled acceptance's noise key
    plant_gap: float = 1.0       # a planted logit is the row maximum + plant_gap

    @property
    def ragged(self) -> bool:
        return self.m_cycle is not None or self.budget >= 0

    def m_req(self) -> torch.Tensor:
        """int32 [B]: lattice positions request b drafts from."""
        cyc = self.m_cycle or (self.m,)
        return torch.tensor([cyc[b % len(cyc)] for b in range(self.B)], dtype=torch.int32)

    @property
    def T(self) -> int:
        return self.N + 1

    @property
    def Lmax(self) -> int:
        return self.L + self.headroom

    @property
    def dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.io == "bf16" else torch.float32

    def replace(self, **kw) -> "SpecConfig":
        return dataclasses.replace(self, **kw)


_BIG = dict(Hk=16, Hv=32, dk=128, dv=128, Hq=32, Hkv=8, D=128, V=151936, io="bf16")

CONFIGS = {
    0: SpecConfig("tiny", B=1, m=4, K=4, N=8, Hk=4, Hv=4, dk=64, dv=64, Hq=4, Hkv=4, D=64,
                  L=128, V=1024, p_plant=0.8, io="f32"),
    1: SpecConfig("single", B=1, m=8, K=16, N=24, L=4096, p_plant=0.85, **_BIG),
    2: SpecConfig("long", B=1, m=16, K=16, N=64, L=16384, p_plant=0.9, **_BIG),
    3: SpecConfig("batched", B=24, m=8, K=16, N=24, L=8192, L_lo=1024, p_plant=0.85, **_BIG),
    4: SpecConfig("stack", B=8, m=8, K=16, N=24, L=8192, p_plant=0.85, n_gdn=48, n_attn=16,
                  **_BIG),
    # batch sharing a 192-node budget, 16/12/8 draft positions per request
    5: SpecConfig("ragged", B=24, m=16, K=16, N=24, L=8192, L_lo=1024, p_plant=0.85,
                  m_cycle=(16, 12, 8), budget=192, **_BIG),
    # 'single' drafted by a drafter with a Markov head (parent-dependent edges)
    6: SpecConfig("markov", B=1, m=8, K=16, N=24, L=4096, p_plant=0.85, markov_R=32, **_BIG),
    # 'single' verified by sampling at temperature 1 (planted tokens carry ~0.88
    # of the target's probability)
    7: SpecConfig("sampled", B=1, m=8, K=16, N=24, L=4096, p_plant=0.85, temperature=1.0,
                  sample_seed=0x5EED_0F_7EE5, plant_gap=10.0, **_BIG),
}


def config(i_or_name) -> SpecConfig:
    if isinstance(i_or_name, SpecConfig):
        return i_or_name
    if isinstance(i_or_name, int):
        return CONFIGS[i_or_name]
    for c in CONFIGS.values():
        if c.name == i_or_name:
            return c
    raise KeyError(i_or_name)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_lattice(cfg: SpecConfig, gen: torch.Generator):
    """Drafter lattice: tokens int32 [B][m][K], scores f32 [B][m][K], root int32 [B]."""
    toks = torch.empty((cfg.B, cfg.m, cfg.K), dtype=torch.int32)
    for b in range(cfg.B):
        for s in range(cfg.m):
            toks[b, s] = torch.randperm(cfg.V, generator=gen)[: cfg.K].to(torch.int32)
    z = torch.randn((cfg.B, cfg.m, cfg.K), generator=gen, dtype=torch.float32) * 2.0
    scores = torch.log_softmax(z, dim=-1).contiguous()
    root = torch.randint(0, cfg.V, (cfg.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    return toks, scores, root


def _unit_rows(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    x = x / x.norm(dim=-1, keepdim=True)
    return x.to(dtype).contiguous()


def make_gdn_layer(cfg: SpecConfig, gen: torch.Generator, device="cpu", batch=None, rows=None):
    """One GDN layer's inputs for every tree row (see module docstring)."""
    B = cfg.B if batch is None else batch
    T = cfg.T if rows is None else rows
    f32 = torch.float32
    kw = dict(generator=gen, device=device, dtype=f32)
    h0 = (torch.randn((B, cfg.Hv, cfg.dk, cfg.dv), **kw) * 0.1).contiguous()
    q = _unit_rows(torch.randn((B, T, cfg.Hk, cfg.dk), **kw), cfg.dtype)
    k = _unit_rows(torch.randn((B, T, cfg.Hk, cfg.dk), **kw), cfg.dtype)
    v = torch.randn((B, T, cfg.Hv, cfg.dv), **kw).to(cfg.dtype).contiguous()
    beta = torch.sigmoid(torch.randn((B, T, cfg.Hv), **kw)).contiguous()
    alpha = (0.9 + 0.1 * torch.rand((B, T, cfg.Hv), **kw)).contiguous()
    return dict(h0=h0, q=q, k=k, v=v, alpha=alpha, beta=beta)


def make_attn_layer(cfg: SpecConfig, gen: torch.Generator, device="cpu", batch=None, rows=None,
                    Lmax=None):
    """One attention layer's tree rows and KV cache (all ~ N(0, 1))."""
    B = cfg.B if batch is None else batch
    T = cfg.T if rows is None else rows
    Lm = cfg.Lmax if Lmax is None else Lmax
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    dt = cfg.dtype
    q = torch.randn((B, T, cfg.Hq, cfg.D), **kw).to(dt).contiguous()
    k_tree = torch.randn((B, T, cfg.Hkv, cfg.D), **kw).to(dt).contiguous()
    v_tree = torch.randn((B, T, cfg.Hkv, cfg.D), **kw).to(dt).contiguous()
    k_cache = torch.randn((B, Lm, cfg.Hkv, cfg.D), **kw).to(dt).contiguous()
    v_cache = torch.randn((B, Lm, cfg.Hkv, cfg.D), **kw).to(dt).contiguous()
    return dict(q=q, k_tree=k_tree, v_tree=v_tree, k_cache=k_cache, v_cache=v_cache)


def make_markov(cfg: SpecConfig, gen: torch.Generator, R: int = 32):
    """Inputs of a drafter with a Markov head: per-candidate base logits
    ~ N(0, 2^2) [B][m][K] (the logits whose log-softmax is the plain lattice's
    score) and the two embedding tables W1, W2 [V][R] ~ N(0, R^-1/2), so the
    Markov term <W1[x], W2[y]> has unit variance."""
    base = (torch.randn((cfg.B, cfg.m, cfg.K), generator=gen) * 2.0).float().contiguous()
    sd = R ** -0.25 if R > 0 else 1.0
    W1 = (torch.randn((cfg.V, R), generator=gen) * sd).float().contiguous()
    W2 = (torch.randn((cfg.V, R), generator=gen) * sd).float().contiguous()
    return base, W1, W2


def make_kv_len(cfg: SpecConfig, gen: torch.Generator) -> torch.Tensor:
    if cfg.L_lo is None:
        return torch.full((cfg.B,), cfg.L, dtype=torch.int32)
    return torch.randint(cfg.L_lo, cfg.L + 1, (cfg.B,), generator=gen,
                         dtype=torch.int64).to(torch.int32)


def make_logits(cfg: SpecConfig, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """Unplanted target logits [B][T][V] ~ N(0, 1) in the I/O type."""
    x = torch.randn((cfg.B, cfg.T, cfg.V), generator=gen, device=device, dtype=torch.float32)
    return x.to(cfg.dtype).contiguous()


def top_candidates(lat_tok: torch.Tensor, lat_score: torch.Tensor) -> torch.Tensor:
    """Token of the highest-scoring candidate of every position, [B][m]
    (first index among equal scores)."""
    best = torch.argmax(lat_score, dim=-1, keepdim=True)
    return torch.gather(lat_tok, -1, best).squeeze(-1)


def first_child_tokens(node_parent, node_rank, node_tok, n_nodes) -> torch.Tensor:
    """[B][T] token of each row's rank-0 child in the tree, -1 where that child
    is not in the tree (indexing only)."""
    par = torch.as_tensor(node_parent).long()
    rank = torch.as_tensor(node_rank).long()
    tok = torch.as_tensor(node_tok).long()
    B, T = par.shape
    out = torch.full((B, T), -1, dtype=torch.long)
    nn = torch.as_tensor(n_nodes).long()
    for b in range(B):
        for x in range(1, int(nn[b])):
            if int(rank[b, x]) == 0:
                out[b, par[b, x]] = tok[b, x]
    return out


def plant_logits(logits: torch.Tensor, lat_tok, lat_score, node_depth, n_nodes, p: float,
                 gen: torch.Generator, first_child=None, gap: float = 1.0) -> torch.Tensor:
    """Plant the drafter's first choice as the argmax of tree rows (in place).

    node_depth [B][T] and n_nodes [B] describe the tree the logits belong to.
    One uniform draw per row decides, independently, whether that row is
    planted (rows of depth m and padding rows never are).  The first choice is
    the top candidate of the next lattice position, or, with first_child
    ([B][T] from first_child_tokens: for drafters whose ranking depends on the
    parent), the row's rank-0 child in the tree (no plant where it is absent).
    The planted logit is the row maximum + gap.
    """
    B, T, V = logits.shape
    m = lat_tok.shape[1]
    dev = logits.device
    u = torch.rand((B, T), generator=gen, dtype=torch.float32, device=gen.device).to(dev)
    depth = torch.as_tensor(node_depth, device=dev).long()
    nn = torch.as_tensor(n_nodes, device=dev).long()
    rows = torch.arange(T, device=dev).unsqueeze(0)
    ok = (u < p) & (rows < nn.unsqueeze(1)) & (depth >= 0) & (depth < m)
    if first_child is None:
        top = top_candidates(torch.as_tensor(lat_tok).to(dev), torch.as_tensor(lat_score).to(dev))
        tok = torch.gather(top.long(), 1, depth.clamp(0, m - 1))
    else:
        tok = torch.as_tensor(first_child).long().to(dev)
        ok = ok & (tok >= 0)
        tok = tok.clamp(min=0)
    val = (logits.float().amax(dim=-1) + gap).to(logits.dtype)
    bi, ti = torch.nonzero(ok, as_tuple=True)
    logits[bi, ti, tok[bi, ti]] = val[bi, ti]
    return logits


# ----------------------------------------------------------- per-token rows

def row_generator(*key) -> torch.Generator:
    """Generator seeded from a tuple such as (seed, layer, request, position,
    token), so that a token's inputs do not depend on the tree it sits in."""
    h = hashlib.sha256(repr(tuple(int(x) for x in key)).encode()).digest()
    return _gen(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))


def fill_rows_by_token(cfg: SpecConfig, seed: int, node_tok, node_depth, n_nodes, kv_len,
                       gdn_layers, attn_layers):
    """Overwrite every tree row's per-token inputs (GDN q/k/v/alpha/beta and
    attention q/k/v) with values drawn from (seed, layer, request, absolute
    position, token); absolute position = kv_len[b] + depth.  Used by the
    multi-step decode-consistency checks."""
    node_tok = torch.as_tensor(node_tok)
    node_depth = torch.as_tensor(node_depth)
    n_nodes = torch.as_tensor(n_nodes)
    kv_len = torch.as_tensor(kv_len)
    for b in range(node_tok.shape[0]):
        for n in range(int(n_nodes[b])):
            pos = int(kv_len[b]) + int(node_depth[b, n])
            tok = int(node_tok[b, n])
            for li, lay in enumerate(gdn_layers):
                g = row_generator(seed, 0, li, b, pos, tok)
                kq = torch.randn((2, cfg.Hk, cfg.dk), generator=g)
                kq = kq / kq.norm(dim=-1, keepdim=True)
                lay["q"][b, n] = kq[0].to(lay["q"].dtype)
                lay["k"][b, n] = kq[1].to(lay["k"].dtype)
                lay["v"][b, n] = torch.randn((cfg.Hv, cfg.dv), generator=g).to(lay["v"].dtype)
                lay["beta"][b, n] = torch.sigmoid(torch.randn((cfg.Hv,), generator=g))
                lay["alpha"][b, n] = 0.9 + 0.1 * torch.rand((cfg.Hv,), generator=g)
            for li, lay in enumerate(attn_layers):
                g = row_generator(seed, 1, li, b, pos, tok)
                lay["q"][b, n] = torch.randn((cfg.Hq, cfg.D), generator=g).to(lay["q"].dtype)
                lay["k_tree"][b, n] = torch.randn((cfg.Hkv, cfg.D), generator=g).to(lay["k_tree"].dtype)
                lay["v_tree"][b, n] = torch.randn((cfg.Hkv, cfg.D), generator=g).to(lay["v_tree"].dtype)


def make_step_inputs(cfg: SpecConfig, seed: int, device="cpu", logits=True) -> dict:
    """All inputs of one verify step except the planted logits (which need the
    tree): lattice, root token, kv_len, n_gdn GDN layers and n_attn attention
    layers, plus unplanted logits when ``logits`` is true.  Everything is drawn
    on the CPU from one generator seeded with ``seed`` and then moved."""
    g = _gen(seed)
    lat_tok, lat_score, root = make_lattice(cfg, g)
    kv_len = make_kv_len(cfg, g)
    gdn = [make_gdn_layer(cfg, g) for _ in range(cfg.n_gdn)]
    attn = [make_attn_layer(cfg, g) for _ in range(cfg.n_attn)]
    out = dict(cfg=cfg, seed=seed, lat_tok=lat_tok, lat_score=lat_score, root_tok=root,
               kv_len=kv_len, gdn=gdn, attn=attn)
    if cfg.ragged:
        out["m_req"] = cfg.m_req()
    if cfg.markov_R > 0:
        out["lat_base"], out["W1"], out["W2"] = make_markov(cfg, g, cfg.markov_R)
    if logits:
        out["logits"] = make_logits(cfg, g)
    out["plant_gen"] = g
    if device != "cpu":
        out = to_device(out, device)
    return out


def to_device(x, device):
    if isinstance(x, torch.Tensor):
        return x.to(device)
    if isinstance(x, dict):
        return {k: to_device(v, device) for k, v in x.items()}
    if isinstance(x, list):
        return [to_device(v, device) for v in x]
    return x
