"""One speculation round over a multi-layer KV cache (attention and sampling only).

MagicDec notes, appendix A.1: the static compressed KV is built at prefill and
reused by every draft step; "Wann beschleunigt spekulatives Decoding das
LLM-Serving?", "Eine Verifizierungsrunde verstehen": gamma draft tokens are
proposed, then the target scores every candidate position in one pass,
modified rejection sampling accepts left to right, and the candidates after
the first rejection are discarded.  With no model weights in scope, a round
here is the sequence of library calls a real round makes, layer by layer, on
synthetic per-layer queries:

    for s in 0 .. gamma-1:
        for layer in 0 .. L-1: draft attention over that layer's compacted cache
        draft-token draw for position s
    for layer in 0 .. L-1: verify attention (gamma+1 rows) over the full cache
    rejection sampling -> out_tokens, num_accepted
    for layer in 0 .. L-1: commit / rollback: keep the accepted verify rows,
        roll back the rest, append the kept rows to the draft cache

Each layer keeps its own kv_len and draft_len arrays (rows [layer, 0] and
[layer, 1] of one int32 buffer), which the commit updates in place, so the
next round reads the committed state.  The per-layer SnapKV draft caches are
selected once in ``prepare()`` (not part of the round), with room for the rows
later rounds append.  ``capture()`` records the round in a CUDA graph; with
``restore=True`` the graph starts by copying the lengths back to their state
after ``prepare()`` (one device-to-device copy), so every replay does the same
work (what the benchmark times).
"""
import torch

from . import mgd, ops
from . import workloads as wl


class SpeculationRound:
    def __init__(self, cfg, device, seed=0, layers=None):
        self.cfg = cfg
        self.dev = device
        self.seed = seed
        self.layers = cfg.get("layers", 1) if layers is None else layers
        self.B, self.Hq, self.Hkv, self.D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
        self.gamma, self.K, self.W, self.P, self.V = cfg["gamma"], cfg["K"], cfg["W"], cfg["pool"], cfg["V"]
        self.T = self.gamma + 1
        self.kv_len = wl.lengths(cfg, seed)
        self.kv_len_d = self.kv_len.to(device)
        self.cap = wl.capacity(cfg, seed)
        self.graph = None

    def prepare(self, spare_rounds=8):
        """Draw every layer's cache and queries and select its draft cache (untimed).  The draft
        caches hold K rows plus room for `spare_rounds` rounds of committed rows."""
        c, dev, B, Hq, Hkv, D, K = self.cfg, self.dev, self.B, self.Hq, self.Hkv, self.D, self.K
        self.k, self.v, self.q, self.qd, self.sel = [], [], [], [], []
        self.draft_cap = K + spare_rounds * self.T
        # lengths[layer, 0] = kv_len, lengths[layer, 1] = draft_len of that layer
        self.lengths = torch.zeros((self.layers, 2, B), dtype=torch.int32, device=dev)
        self.lengths[:, 0] = self.kv_len_d
        ws_snap = ops.workspace(mgd.mgd_snapkv_workspace_size(B, Hq, Hkv, D, self.cap, self.W), dev)
        i32 = torch.int32
        for layer in range(self.layers):
            k, v = wl.kv_cache(c, dev, self.seed, layer=layer, kv_len=self.kv_len, cap=self.cap)
            qw = wl.window_queries(c, dev, self.seed, layer=layer)
            sel = dict(sel_idx=torch.empty((B, Hkv, self.draft_cap), dtype=i32, device=dev),
                       k_draft=torch.zeros((B, Hkv, self.draft_cap, D), dtype=k.dtype, device=dev),
                       v_draft=torch.zeros((B, Hkv, self.draft_cap, D), dtype=k.dtype, device=dev),
                       draft_len=self.lengths[layer, 1], scores=None)
            self.sel.append(ops.snapkv_select(qw, k, v, self.lengths[layer, 0], self.W, self.P, K,
                                              draft_cap=self.draft_cap, ws=ws_snap, out=sel))
            self.k.append(k)
            self.v.append(v)
            self.q.append(wl.queries(c, dev, self.seed, layer=layer))
            self.qd.append(torch.stack([wl.draft_queries(c, dev, self.seed, layer=layer, step=s)[:, 0]
                                        for s in range(self.gamma)]))
            del qw
        del ws_snap
        self.t, self.d = wl.logits(c, dev, self.seed)
        self.u = wl.uniforms(c, dev, self.seed)
        f32, i32 = torch.float32, torch.int32
        self.dout = torch.empty((self.layers, self.gamma, B, Hq, D), dtype=f32, device=dev)
        self.dlse = torch.empty((B, Hq), dtype=f32, device=dev)
        self.vout = torch.empty((self.layers, B, self.T, Hq, D), dtype=f32, device=dev)
        self.vlse = torch.empty((B, self.T, Hq), dtype=f32, device=dev)
        self.tok = torch.empty((B, self.gamma), dtype=i32, device=dev)
        self.out_tok = torch.empty((B, self.T), dtype=i32, device=dev)
        self.nacc = torch.empty((B,), dtype=i32, device=dev)
        self.ws_draft = ops.workspace(mgd.mgd_draft_workspace_size(B, Hq, Hkv, D, self.draft_cap), dev)
        self.ws_verify = ops.workspace(mgd.mgd_verify_workspace_size(B, self.T, Hq, Hkv, D, self.cap), dev)
        self.ws_spec = ops.workspace(mgd.mgd_spec_workspace_size(B, self.gamma, self.V), dev)
        self.ws_commit = ops.workspace(mgd.mgd_commit_workspace_size(B), dev)
        torch.cuda.synchronize(dev)
        self.lengths0 = self.lengths.clone()  # the state every restored round starts from
        esz = 2
        L = self.kv_len.double()
        self.bytes_verify = float((2 * Hkv * L * D * esz).sum()) * self.layers
        self.bytes_draft = float((2 * Hkv * torch.clamp(L, max=K) * D * esz).sum()) * self.layers * self.gamma
        return self

    @property
    def launches(self):
        """Kernels of this library launched per round: gamma x (one draft attention per layer + one
        one-row draw), one verify per layer, rejection sampling (2 kernels), one commit per layer."""
        return self.gamma * self.layers + self.gamma + self.layers + 2 + self.layers

    def propose(self):
        """The draft phase: gamma x (draft attention over every layer's compacted cache, one draw)."""
        for s in range(self.gamma):
            for layer in range(self.layers):
                sel = self.sel[layer]
                ops.draft_attn(self.qd[layer][s], sel["k_draft"], sel["v_draft"], self.lengths[layer, 1],
                               ws=self.ws_draft, out=self.dout[layer, s], lse=self.dlse)
            ops.draft_draw(self.d, self.u, draft_tokens=self.tok, row=s, ws=self.ws_spec)

    def verify_and_sample(self):
        """Verify attention over every layer's full cache, then rejection sampling."""
        for layer in range(self.layers):
            ops.verify_attn(self.q[layer], self.k[layer], self.v[layer], self.lengths[layer, 0], ws=self.ws_verify,
                            out=self.vout[layer], lse=self.vlse)
        ops.rejection_sample(self.t, self.d, self.tok, self.u, ws=self.ws_spec, out_tokens=self.out_tok,
                             num_accepted=self.nacc, reuse_draft_stats=True)

    def commit(self):
        """Commit / rollback of every layer's caches after the round's acceptance decisions."""
        for layer in range(self.layers):
            sel = self.sel[layer]
            ops.commit_round(self.nacc, self.gamma, self.lengths[layer, 0], self.k[layer], self.v[layer],
                             sel["k_draft"], sel["v_draft"], self.lengths[layer, 1], ws=self.ws_commit)

    def restore(self):
        """Lengths back to their state after prepare() (one device copy)."""
        self.lengths.copy_(self.lengths0)

    def run(self):
        self.propose()
        self.verify_and_sample()
        self.commit()

    def _graph_of(self, fn):
        fn()  # eager warm-up
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def capture(self, restore=False):
        """Record one round in a CUDA graph (after an eager warm-up run); with restore=True the
        graph first puts the lengths back to their state after prepare()."""
        def one():
            if restore:
                self.restore()
            self.run()
        self.graph = self._graph_of(one)
        self.restore()
        return self.graph

    def capture_phases(self):
        """Record the phases of a restored round in graphs of their own, for timing each: the
        proposal, the verification and correction, and the commit (which restores first)."""
        def commit():
            self.restore()
            self.commit()
        graphs = [self._graph_of(fn) for fn in (self.propose, self.verify_and_sample, commit)]
        self.restore()
        return graphs

    def replay(self):
        if self.graph is None:
            self.run()
        else:
            self.graph.replay()
