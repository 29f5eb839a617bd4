"""One whole verify step on device buffers: tree build, every GDN layer, every
attention layer, then acceptance and commit -- each a call through the C ABI.

The driver owns the device buffers (stacked per layer, layer outermost, so
the commit sees every layer through one pointer per tensor) and issues the
calls on one stream.  It does no arithmetic of its own.
"""
from __future__ import annotations

import torch

from . import binding
from .synth import SpecConfig


def stack_inputs(inp: dict, device="cuda") -> dict:
    """Device copies of synth.make_step_inputs' output with layers stacked."""
    d = {}
    for k in ("lat_tok", "lat_score", "root_tok", "kv_len", "logits", "m_req", "lat_base", "W1",
              "W2"):
        if k in inp:
            d[k] = inp[k].to(device).contiguous()
    g, a = inp["gdn"], inp["attn"]
    for src, dst in (("h0", "gdn_h0"), ("q", "gdn_q"), ("k", "gdn_k"), ("v", "gdn_v"),
                     ("alpha", "gdn_alpha"), ("beta", "gdn_beta")):
        d[dst] = torch.stack([lay[src] for lay in g]).to(device).contiguous() if g else None
    for src, dst in (("q", "attn_q"), ("k_tree", "k_tree"), ("v_tree", "v_tree"),
                     ("k_cache", "k_cache"), ("v_cache", "v_cache")):
        d[dst] = torch.stack([lay[src] for lay in a]).to(device).contiguous() if a else None
    return d


class VerifyStep:
    """Buffers and calls of one verify step for a synthetic workload."""

    def __init__(self, scfg: SpecConfig, x: dict, device="cuda", persistent: bool = False):
        self.scfg = scfg
        self.persistent = persistent
        self.cfg = binding.make_cfg(scfg)
        self.x = x
        self.device = device
        c = self.cfg
        T = c.N + 1
        dt = torch.bfloat16 if scfg.io == "bf16" else torch.float32
        self.tree = binding.TreeBuffers(c, device)
        self.acc = binding.AcceptBuffers(c, device)
        self.ws = binding.alloc_workspace(c, device)
        self.gdn_o = torch.empty((c.n_gdn_layers, c.B, T, c.Hv, c.dv), dtype=dt, device=device)
        self.attn_o = torch.empty((c.n_attn_layers, c.B, T, c.Hq, c.D), dtype=dt, device=device)

    # the three phases ----------------------------------------------------------
    def build_tree(self, stream=None):
        x = self.x
        if self.scfg.markov_R > 0:
            binding.spec_tree_build_markov(self.cfg, x["lat_tok"], x["lat_base"], x["W1"], x["W2"],
                                           x["root_tok"], self.tree, self.ws, stream)
        elif self.scfg.ragged:
            binding.spec_tree_build_ragged(self.cfg, x["lat_tok"], x["lat_score"], x["root_tok"],
                                           x.get("m_req"), self.scfg.budget, self.tree, self.ws,
                                           stream)
        else:
            binding.spec_tree_build(self.cfg, x["lat_tok"], x["lat_score"], x["root_tok"],
                                    self.tree, self.ws, stream)

    def verify_gdn(self, stream=None):
        x, c = self.x, self.cfg
        for l in range(c.n_gdn_layers):
            binding.gdn_tree_verify(c, self.tree, x["gdn_h0"][l], x["gdn_q"][l], x["gdn_k"][l],
                                    x["gdn_v"][l], x["gdn_alpha"][l], x["gdn_beta"][l],
                                    self.gdn_o[l], None, self.ws, stream)

    def verify_attention(self, stream=None):
        x, c = self.x, self.cfg
        for l in range(c.n_attn_layers):
            binding.attn_tree_verify(c, self.tree, x["attn_q"][l], x["k_tree"][l], x["v_tree"][l],
                                     x["k_cache"][l], x["v_cache"][l], x["kv_len"],
                                     self.attn_o[l], self.ws, stream)

    def verify(self, stream=None):
        self.verify_gdn(stream)
        self.verify_attention(stream)

    def commit_io(self) -> dict:
        x = self.x
        return dict(h0=x["gdn_h0"], gdn_k=x["gdn_k"], gdn_v=x["gdn_v"], alpha=x["gdn_alpha"],
                    beta=x["gdn_beta"], k_tree=x["k_tree"], v_tree=x["v_tree"],
                    k_cache=x["k_cache"], v_cache=x["v_cache"], kv_len=x["kv_len"],
                    root_tok=x["root_tok"])

    def accept_commit(self, stream=None):
        if self.scfg.temperature > 0:
            binding.accept_and_commit_sampled(self.cfg, self.tree, self.x["logits"],
                                              self.sampling(), self.commit_io(), self.acc,
                                              self.ws, stream)
        else:
            binding.accept_and_commit(self.cfg, self.tree, self.x["logits"], self.commit_io(),
                                      self.acc, self.ws, stream)

    def sampling(self):
        return binding.sampling(self.scfg.temperature, self.scfg.sample_seed)

    def run_calls(self, stream=None):
        """The step as the four single-operation calls."""
        self.build_tree(stream)
        self.verify(stream)
        self.accept_commit(stream)

    def run(self, stream=None):
        """The step as one spec_verify_step call (programmatic dependent launch)."""
        x = self.x
        step = dict(gdn_q=x["gdn_q"], gdn_o=self.gdn_o if self.cfg.n_gdn_layers else None,
                    gdn_c=None, attn_q=x["attn_q"],
                    attn_o=self.attn_o if self.cfg.n_attn_layers else None)
        if self.persistent:
            if self.scfg.markov_R > 0 or self.scfg.ragged or self.scfg.temperature > 0:
                raise ValueError("the persistent step takes the plain lattice and the argmax")
            binding.spec_verify_step_persistent(self.cfg, x["lat_tok"], x["lat_score"], self.tree,
                                                step, x["logits"], self.commit_io(), self.acc,
                                                self.ws, stream)
        elif self.scfg.temperature > 0:
            if self.scfg.markov_R > 0 or self.scfg.ragged:
                raise ValueError("the fused sampled step takes the plain lattice")
            binding.spec_verify_step_sampled(self.cfg, x["lat_tok"], x["lat_score"],
                                             self.sampling(), self.tree, step, x["logits"],
                                             self.commit_io(), self.acc, self.ws, stream)
        elif self.scfg.markov_R > 0:
            binding.spec_verify_step_markov(self.cfg, x["lat_tok"], x["lat_base"], x["W1"], x["W2"],
                                            self.tree, step, x["logits"], self.commit_io(), self.acc,
                                            self.ws, stream)
        elif self.scfg.ragged:
            binding.spec_verify_step_ragged(self.cfg, x["lat_tok"], x["lat_score"], x.get("m_req"),
                                            self.scfg.budget, self.tree, step, x["logits"],
                                            self.commit_io(), self.acc, self.ws, stream)
        else:
            binding.spec_verify_step(self.cfg, x["lat_tok"], x["lat_score"], self.tree, step,
                                     x["logits"], self.commit_io(), self.acc, self.ws, stream)

    @property
    def launches_per_step(self) -> int:
        if self.persistent:
            return binding.spec_step_launches_persistent(self.cfg)
        # the shared budget adds one launch (the selection) to the step; the
        # sampled acceptance is a launch of its own (the argmax shares the last
        # attention merge's)
        extra = (1 if self.scfg.budget >= 0 else 0)
        merged = self.cfg.n_attn_layers > 0 and self.cfg.B * (self.cfg.N + 1) <= 64
        extra += 1 if (self.scfg.temperature > 0 and merged) else 0
        return binding.spec_step_launches(self.cfg) + extra


# The step's per-step inputs in three pieces, in the order the copies are
# issued: the lattice with the attention rows (the tree build and the
# attention layers), the GDN rows, then the logits, read only by the
# acceptance.  Each copy costs a few microseconds of its own, so small pieces
# go together; the GDN rows stay apart because with many GDN layers they are
# most of the non-logits bytes and the attention need not wait for them.
HOST_PIECES = (("rows", ("lat_tok", "lat_score", "m_req", "lat_base", "attn_q", "k_tree",
                         "v_tree")),
               ("gdn", ("gdn_q", "gdn_k", "gdn_v", "gdn_alpha", "gdn_beta")),
               ("logits", ("logits",)))


class HostStep:
    """A verify step whose per-step inputs come from pinned host memory.

    The inputs are copied in three pieces on a copy stream (the lattice with
    the attention rows, the GDN rows, the logits), in the order the step reads
    them, and each phase on the compute stream waits only for its own piece:
    the logits -- most of the bytes -- are copied while the tree, attention
    and GDN layers run, and only the acceptance and commit wait for them.  The accepted lengths and tokens come back to pinned host
    memory at the end.  The whole sequence is captured once as a CUDA graph
    and replayed per step.

    st: a VerifyStep whose per-step input tensors this object re-points at
    its device pieces (their current values are copied into the pinned host
    buffers, which the caller then refills per step through `views`).
    """

    def __init__(self, st: "VerifyStep"):
        self.st = st
        x = st.x
        self.host, self.dev, self.views = {}, {}, {}
        self.h2d_bytes = 0
        for piece, keys in HOST_PIECES:
            keys = [k for k in keys if x.get(k) is not None]
            if not keys:
                continue
            offs, total = {}, 0
            for k in keys:
                offs[k] = total
                total += (x[k].numel() * x[k].element_size() + 255) // 256 * 256
            dev = torch.empty(total, dtype=torch.uint8, device=st.device)
            host = torch.empty(total, dtype=torch.uint8).pin_memory()
            for k in keys:
                n = x[k].numel() * x[k].element_size()
                view = dev[offs[k]:offs[k] + n].view(x[k].dtype).view(x[k].shape)
                view.copy_(x[k])
                host[offs[k]:offs[k] + n].copy_(x[k].cpu().contiguous().view(-1).view(torch.uint8))
                x[k] = view
                self.views[k] = host[offs[k]:offs[k] + n].view(view.dtype).view(view.shape)
            self.host[piece], self.dev[piece] = host, dev
            self.h2d_bytes += sum(x[k].numel() * x[k].element_size() for k in keys)
        self.out = {k: torch.empty_like(getattr(st.acc, k), device="cpu").pin_memory()
                    for k in ("accept_len", "out_tok")}
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.out.values())
        self.copy_stream = torch.cuda.Stream(device=st.device)
        self.graph = None

    def _sequence(self):
        st = self.st
        comp = torch.cuda.current_stream()
        cs = self.copy_stream
        cs.wait_stream(comp)                 # the previous step's readers are done
        ev = {}
        with torch.cuda.stream(cs):
            for piece, _ in HOST_PIECES:
                if piece in self.dev:
                    self.dev[piece].copy_(self.host[piece], non_blocking=True)
                    ev[piece] = torch.cuda.Event()
                    ev[piece].record(cs)
        for piece, run in (("rows", st.build_tree), (None, st.verify_attention),
                           ("gdn", st.verify_gdn), ("logits", st.accept_commit)):
            if piece in ev:
                comp.wait_event(ev[piece])
            run()
        comp.wait_stream(cs)
        for k, t in self.out.items():
            t.copy_(getattr(st.acc, k), non_blocking=True)

    def capture(self):
        """Run the copies, the four phases and the result read-back once,
        then capture them as a CUDA graph."""
        self._sequence()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            self._sequence()
        torch.cuda.synchronize()

    def run(self):
        """One step: copies in, the step, results out (asynchronous on the
        current stream; synchronize before reading self.out)."""
        if self.graph is None:
            self.capture()
        self.graph.replay()
