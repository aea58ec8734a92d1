"""One QSPEC round as a sequence of library calls that a CUDA graph can hold.

QSPEC summary page, "QSPEC structure": a round runs gamma draft passes in the
W4A4 configuration (every linear of every layer plus the LM head at M = B),
one verify pass in the W4A16 configuration over the gamma + 1 candidate rows
of every sequence (M = B (gamma + 1)), the acceptance decision, and the
overwrite of the accepted rows' KV-cache entries with the verify pass's.

The model operations between the linears (attention, norms, activation
functions, embeddings) are outside this library, so every linear reads its
own seeded activations and the verification reads seeded target / draft
logits: the round issues exactly the hot-path calls of a real round, on
inputs of the real shapes.  All buffers are allocated once here; `run`
only launches kernels (through the C ABI), so a round can be captured into
a CUDA graph and replayed, with the round id (the verification's random
stream) fixed per captured graph.
"""
from __future__ import annotations

import torch

from . import binding as q
from . import synthetic as syn

GROUP = 128


class QspecRound:
    """Buffers and calls of one round.

    shape: a model shape dict (`synthetic.LLAMA3_8B`, `synthetic.QWEN25_7B`
    or one of the same keys); B sequences, gamma drafts per sequence, a KV
    cache of T positions; `seed` fixes every input.  outliers, p_std and
    q_noise shape the synthetic activations and logits (see `synthetic`).
    """

    def __init__(self, shape: dict, B: int, gamma: int, T: int, seed: int, device, outliers=0.0,
                 p_std=3.0, q_noise=0.5):
        dev = torch.device(device)
        self.dev = dev
        self.shape = shape
        self.B, self.gamma, self.T, self.seed = B, gamma, T, seed
        self.L, self.hidden, self.V = shape["layers"], shape["hidden"], shape["vocab"]
        self.H, self.D = shape["kv_heads"], shape["head_dim"]
        self.linears = syn.fused_layer_linears(shape)
        g, L = gamma, self.L
        Mv = B * (g + 1)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # weights: one packed INT4 set per linear, shared by both passes
        self.w = []
        for l in range(L):
            lw = {}
            for j, (name, N, K) in enumerate(self.linears):
                codes, s, z = syn.weights(N, K, self.weight_seed(l, j), device=dev)
                lw[name] = q.pack_weights(codes, s, z, dev_status=self.status)
                del codes, s, z
            self.w.append(lw)
        codes, s, z = syn.weights(self.V, self.hidden, self.weight_seed(-1, 0), device=dev)
        self.lm = q.pack_weights(codes, s, z, dev_status=self.status)
        del codes, s, z
        # inputs: draft activations [gamma][L][B][K] per linear, verify [L][Mv][K]
        self.xd, self.xv = {}, {}
        for j, (name, N, K) in enumerate(self.linears):
            self.xd[name] = syn.activations(g * L * B, K, seed * 7 + j, device=dev,
                                            outlier_frac=outliers).view(g, L, B, K)
            self.xv[name] = syn.activations(L * Mv, K, seed * 11 + j, device=dev,
                                            outlier_frac=outliers).view(L, Mv, K)
        self.xd_lm = syn.activations(g * B, self.hidden, seed * 13, device=dev,
                                     outlier_frac=outliers).view(g, B, self.hidden)
        self.xv_lm = syn.activations(Mv, self.hidden, seed * 17, device=dev, outlier_frac=outliers)
        P, Q, d = syn.logits_noisy_draft(B, g, self.V, seed * 19, device=dev, p_std=p_std,
                                         q_noise=q_noise)
        self.P, self.Q, self.drafts = P, Q, d
        self.kc, self.vc = syn.kv_cache(L, B, self.H, T, self.D, seed * 23, device=dev)
        self.kn, self.vn = syn.kv_new(L, B, g, self.H, self.D, seed * 29, device=dev)
        self.base = syn.base_positions(B, T, g, seed * 31, device=dev)
        # scratch and outputs
        Ks = sorted({K for _, _, K in self.linears} | {self.hidden})
        self.qbuf = {K: (torch.empty((B, K // 2), dtype=torch.uint8, device=dev),
                         torch.empty((B, K // GROUP), dtype=torch.float32, device=dev),
                         torch.empty((B, K // GROUP), dtype=torch.int32, device=dev)) for K in Ks}
        self.yd = {name: torch.empty((B, N), dtype=torch.bfloat16, device=dev)
                   for name, N, _ in self.linears}
        self.yv = {name: torch.empty((Mv, N), dtype=torch.bfloat16, device=dev)
                   for name, N, _ in self.linears}
        self.yd_lm = torch.empty((B, self.V), dtype=torch.bfloat16, device=dev)
        self.yv_lm = torch.empty((Mv, self.V), dtype=torch.bfloat16, device=dev)
        self.ws = q.verify_workspace(B, g, self.V, dev)
        self.n_acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.out = torch.zeros((B, g + 1), dtype=torch.int32, device=dev)
        self.verify_seed = 1234
        torch.cuda.synchronize(dev)

    def weight_seed(self, layer: int, j: int) -> int:
        """Seed of the weights of linear j of a layer (layer -1: the LM head)."""
        return self.seed * 100003 + (7777 if layer < 0 else layer * 8 + j)

    @staticmethod
    def _check(rc, what):
        if rc != 0:
            raise q.QspecError(rc, what)

    def _w4a4(self, x, pk, N, K, y):
        """a2 + a3: quantise the bf16 activations and run the W4A4 linear."""
        xq, sx, qs = self.qbuf[K]
        M = x.shape[0]
        self._check(q.qspec_linear_w4a4_bf16(x, K, pk[0], pk[1], M, N, K, y, N, xq, sx, qs, None,
                                             self.status), "qspec_linear_w4a4_bf16")

    def draft_linears(self, j=0):
        """Draft step j's W4A4 launches (every linear of every layer, then the
        LM head), as the round makes them."""
        for l in range(self.L):
            for name, N, K in self.linears:
                self._w4a4(self.xd[name][j, l], self.w[l][name], N, K, self.yd[name])
        self._w4a4(self.xd_lm[j], self.lm, self.V, self.hidden, self.yd_lm)

    def verify_linears(self):
        """The verify pass's W4A16 launches."""
        Mv = self.B * (self.gamma + 1)
        for l in range(self.L):
            for name, N, K in self.linears:
                self._check(q.qspec_linear_w4a16(self.xv[name][l], K, self.w[l][name][0],
                                                 self.w[l][name][1], Mv, N, K, self.yv[name], N,
                                                 self.status), "qspec_linear_w4a16")
        self._check(q.qspec_linear_w4a16(self.xv_lm, self.hidden, self.lm[0], self.lm[1], Mv,
                                         self.V, self.hidden, self.yv_lm, self.V, self.status),
                    "qspec_linear_w4a16")

    def run(self, rnd: int, acc_slot=None):
        """Launch round `rnd` on the current stream: gamma draft steps, the
        verify pass, sampled verification (round id rnd), the KV overwrite;
        acc_slot (int32 [B], device), if given, receives A_b."""
        for j in range(self.gamma):
            self.draft_linears(j)
        self.verify_linears()
        self._check(q.qspec_verify_sample(self.P, self.Q, self.drafts, self.B, self.gamma, self.V,
                                          self.verify_seed, rnd, self.n_acc, self.out, self.ws,
                                          self.ws.numel(), self.status), "qspec_verify_sample")
        self._check(q.qspec_kv_overwrite(self.kc, self.vc, self.kn, self.vn, self.base, self.n_acc,
                                         self.L, self.B, self.H, self.T, self.D, self.gamma,
                                         self.status), "qspec_kv_overwrite")
        if acc_slot is not None:
            acc_slot.copy_(self.n_acc, non_blocking=True)

    def capture(self, rnd: int, stream: torch.cuda.Stream, acc_slot=None) -> torch.cuda.CUDAGraph:
        """Round `rnd` captured into a CUDA graph on `stream` (run one round
        eagerly first: the first call of each kernel sets its attributes)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run(rnd, acc_slot)
        return g

    def host_inputs(self):
        """The tensors a round reads from outside: all activations, logits,
        drafts and cache positions (weights and the cache stay resident)."""
        t = [self.xd[n] for n, _, _ in self.linears] + [self.xv[n] for n, _, _ in self.linears]
        return t + [self.xd_lm, self.xv_lm, self.P, self.Q, self.drafts, self.base]

    def device_status(self) -> int:
        torch.cuda.synchronize(self.dev)
        return int(self.status.item())
