"""One speculation round over a multi-layer KV cache (attention and sampling only).

MagicDec notes, appendix A.1: the static compressed KV is built at prefill and
reused by every draft step; "Wann beschleunigt spekulatives Decoding das
LLM-Serving?", "Eine Verifizierungsrunde verstehen": gamma draft tokens are
proposed, then the target scores every candidate position in one pass and
modified rejection sampling accepts left to right.  With no model weights in
scope, a round here is the sequence of library calls a real round makes,
layer by layer, on synthetic per-layer queries:

    for s in 0 .. gamma-1:
        for layer in 0 .. L-1: draft attention over that layer's compacted cache
        draft-token draw for position s
    for layer in 0 .. L-1: verify attention (gamma+1 rows) over the full cache
    rejection sampling -> out_tokens, num_accepted

The per-layer SnapKV draft caches are selected once in ``prepare()`` (not
part of the round).  ``capture()`` records the round in a CUDA graph so the
(gamma+1)*L + gamma + 2 kernel launches replay without host overhead.
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

    def prepare(self):
        """Draw every layer's cache and queries and select its draft cache (untimed)."""
        c, dev, B, Hq, Hkv, D, K = self.cfg, self.dev, self.B, self.Hq, self.Hkv, self.D, self.K
        self.k, self.v, self.q, self.qd, self.sel = [], [], [], [], []
        ws_snap = ops.workspace(mgd.mgd_snapkv_workspace_size(B, Hq, Hkv, D, self.cap, self.W), dev)
        for layer in range(self.layers):
            k, v = wl.kv_cache(c, dev, self.seed, layer=layer, kv_len=self.kv_len, cap=self.cap)
            qw = wl.window_queries(c, dev, self.seed, layer=layer)
            self.sel.append(ops.snapkv_select(qw, k, v, self.kv_len_d, self.W, self.P, K, ws=ws_snap))
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
        self.ws_draft = ops.workspace(mgd.mgd_draft_workspace_size(B, Hq, Hkv, D, K), dev)
        self.ws_verify = ops.workspace(mgd.mgd_verify_workspace_size(B, self.T, Hq, Hkv, D, self.cap), dev)
        self.ws_spec = ops.workspace(mgd.mgd_spec_workspace_size(B, self.gamma, self.V), dev)
        esz = 2
        L = self.kv_len.double()
        self.bytes_verify = float((2 * Hkv * L * D * esz).sum()) * self.layers
        self.bytes_draft = float((2 * Hkv * torch.clamp(L, max=K) * D * esz).sum()) * self.layers * self.gamma
        return self

    @property
    def launches(self):
        """Kernels of this library launched per round."""
        return self.gamma * self.layers + self.gamma + self.layers + 2  # one-row draws: 1 kernel; sampling: 2

    def propose(self):
        """The draft phase: gamma x (draft attention over every layer's compacted cache, one draw)."""
        for s in range(self.gamma):
            for layer in range(self.layers):
                sel = self.sel[layer]
                ops.draft_attn(self.qd[layer][s], sel["k_draft"], sel["v_draft"], sel["draft_len"],
                               ws=self.ws_draft, out=self.dout[layer, s], lse=self.dlse)
            ops.draft_draw(self.d, self.u, draft_tokens=self.tok, row=s, ws=self.ws_spec)

    def verify_and_sample(self):
        """Verify attention over every layer's full cache, then rejection sampling."""
        for layer in range(self.layers):
            ops.verify_attn(self.q[layer], self.k[layer], self.v[layer], self.kv_len_d, ws=self.ws_verify,
                            out=self.vout[layer], lse=self.vlse)
        ops.rejection_sample(self.t, self.d, self.tok, self.u, ws=self.ws_spec, out_tokens=self.out_tok,
                             num_accepted=self.nacc)

    def run(self):
        self.propose()
        self.verify_and_sample()

    def capture(self):
        """Record one round in a CUDA graph (after an eager warm-up run)."""
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def capture_phases(self):
        """Record the two phases of a round in graphs of their own, for timing each."""
        graphs = []
        for fn in (self.propose, self.verify_and_sample):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs.append(g)
        return graphs

    def replay(self):
        if self.graph is None:
            self.run()
        else:
            self.graph.replay()
