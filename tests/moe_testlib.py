"""Shared helpers for the parity tests: build seeded problems, run the CUDA
path step by step through the C-ABI binding, and evaluate the oracle on the
same bytes."""

import numpy as np
import torch

import oracle
import synth


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def bf16_to_f64(t):
    # whole stage buffers come through here, and their padding rows are left
    # unwritten by design: a signalling NaN pattern there is not an error
    with np.errstate(invalid="ignore"):
        return t.detach().float().cpu().numpy().astype(np.float64)


class Problem:
    """Seeded inputs of one layer shape (CPU copies + device copies)."""

    def __init__(self, T, K, I, E_global, E_local, topk, dtype, layout="auto", expert_start=0, max_m=0,
                 seed=1, zipf_s=None, drop_every=0, weight_device="cuda", weight_seed=None):
        self.T, self.K, self.I = T, K, I
        self.E_global, self.E_local, self.topk = E_global, E_local, topk
        self.dtype, self.expert_start = dtype, expert_start
        if layout == "auto":
            layout = "masked" if oracle.use_masked_layout(E_global, E_local) else "compact"
        self.layout = layout
        self.max_m = max_m if max_m else (T if layout == "masked" else 0)
        if layout == "masked" and self.max_m < max(T, 1):
            self.max_m = max(T, 1)
        self.x = synth.activations(T, K, seed)
        ids, w = synth.routing(T, E_global, topk, seed + 1, zipf_s)
        if drop_every:
            ids[::drop_every, -1] = -1
        self.ids, self.w = ids, w
        ws = seed + 2 if weight_seed is None else weight_seed
        if dtype == "fp8":
            self.w13, self.w13_sf = synth.fp8_expert_weights(E_local, 2 * I, K, ws, weight_device, expert_start)
            self.w2, self.w2_sf = synth.fp8_expert_weights(E_local, K, I, ws + 1, weight_device, expert_start)
        elif dtype == "mxfp4":
            # packed E2M1 codes + natural [E, N, C/32] scales; GpuLayer packs the scales
            self.w13, self.w13_sf = synth.mxfp4_expert_weights(E_local, 2 * I, K, ws, weight_device, expert_start)
            self.w2, self.w2_sf = synth.mxfp4_expert_weights(E_local, K, I, ws + 1, weight_device, expert_start)
        elif dtype == "mxfp8":
            # natural [E, N, C/32] scale layout; GpuLayer packs it for the device
            self.w13, self.w13_sf = synth.mxfp8_expert_weights(E_local, 2 * I, K, ws, weight_device, expert_start)
            self.w2, self.w2_sf = synth.mxfp8_expert_weights(E_local, K, I, ws + 1, weight_device, expert_start)
        else:
            self.w13 = synth.bf16_expert_weights(E_local, 2 * I, K, ws, weight_device, expert_start)
            self.w2 = synth.bf16_expert_weights(E_local, K, I, ws + 1, weight_device, expert_start)
            self.w13_sf = self.w2_sf = None
        self._deq = {}

    # ----------------------------------------------------------------- oracle side
    def x64(self):
        return bf16_to_f64(self.x)

    def expert_weights64(self, e):
        """fp64 dequantised (w13[e], w2[e]) for local expert e (cached)."""
        if e not in self._deq:
            if self.dtype in ("fp8", "mxfp8", "mxfp4"):
                deq = {"fp8": oracle.dequant_fp8_weights, "mxfp8": oracle.dequant_mx_weights,
                       "mxfp4": oracle.dequant_mxfp4_weights}[self.dtype]
                w13 = deq(self.w13[e:e + 1].cpu().numpy(), self.w13_sf[e:e + 1].cpu().numpy().astype(np.int64) - 127)[0]
                w2 = deq(self.w2[e:e + 1].cpu().numpy(), self.w2_sf[e:e + 1].cpu().numpy().astype(np.int64) - 127)[0]
            else:
                w13 = bf16_to_f64(self.w13[e])
                w2 = bf16_to_f64(self.w2[e])
            self._deq[e] = (w13, w2)
        return self._deq[e]

    def all_weights64(self):
        pairs = [self.expert_weights64(e) for e in range(self.E_local)]
        return np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])

    def oracle_plan(self):
        return oracle.plan_layout(self.ids.numpy(), self.E_global, self.E_local, self.expert_start, self.layout,
                                  128, self.max_m if self.layout == "masked" else None)

    def oracle_forward(self, keep=False):
        w13, w2 = self.all_weights64()
        return oracle.forward_layout(self.x64(), w13, w2, self.ids.numpy(), self.w.numpy(), self.dtype,
                                     self.E_global, self.expert_start, layout=self.layout,
                                     max_m=self.max_m if self.layout == "masked" else None, keep=keep)

    def oracle_tokens(self, tokens):
        """Output rows of the given tokens by the per-token oracle (only the
        experts those tokens use are dequantised)."""
        out = []
        x = self.x64()
        for t in tokens:
            ids = self.ids[t].numpy()
            loc = [int(i) - self.expert_start for i in ids
                   if 0 <= int(i) < self.E_global and 0 <= int(i) - self.expert_start < self.E_local]
            uniq = sorted(set(loc))
            if not uniq:
                out.append(np.zeros(self.K))
                continue
            w13 = np.stack([self.expert_weights64(e)[0] for e in uniq])
            w2 = np.stack([self.expert_weights64(e)[1] for e in uniq])
            remap = np.array([[uniq.index(int(i) - self.expert_start)
                               if 0 <= int(i) < self.E_global and 0 <= int(i) - self.expert_start < self.E_local
                               else -1 for i in ids]])
            out.append(oracle.forward_per_token(x[t:t + 1], w13, w2, remap, self.w[t:t + 1].numpy(), self.dtype,
                                                E_global=len(uniq), expert_start=0)[0])
        return np.stack(out)

    # ----------------------------------------------------------------- CUDA side
    def gpu(self):
        return GpuLayer(self)


class GpuLayer:
    def __init__(self, p):
        import moe_expert_layer_ep_gb300 as M
        self.M, self.p = M, p
        self.shape = M.make_shape(p.T, p.K, p.I, p.E_global, p.E_local, p.topk, p.dtype, p.layout,
                                  p.expert_start, p.max_m)
        dev = "cuda"
        self.w13 = p.w13.to(dev)
        self.w2 = p.w2.to(dev)
        self.w13_sf = None if p.w13_sf is None else p.w13_sf.to(dev)
        self.w2_sf = None if p.w2_sf is None else p.w2_sf.to(dev)
        if p.dtype in ("mxfp8", "mxfp4"):
            self.w13_sf = M.moe_pack_mx_scales(self.w13_sf)
            self.w2_sf = M.moe_pack_mx_scales(self.w2_sf)
        self.ctx = M.moe_ctx_create(self.shape, self.w13, self.w13_sf, self.w2, self.w2_sf)
        self.ws = M.alloc_workspace(self.ctx)
        self.x = p.x.to(dev)
        self.ids = p.ids.to(dev)
        self.w = p.w.to(dev)
        self.out = torch.empty((p.T, p.K), dtype=torch.bfloat16, device=dev)
        M.moe_clear_device_status(self.ws)

    def view(self, name):
        return self.M.ws_view(self.ctx, self.ws, name)

    def plan(self):
        self.M.moe_plan_layout(self.ctx, self.ids, self.ws)

    def quant(self):
        self.M.moe_quant_scatter(self.ctx, self.x, self.ws)

    def gemm1(self):
        self.M.moe_grouped_gemm_w13_act(self.ctx, self.ws)

    def gemm2(self):
        self.M.moe_grouped_gemm_w2(self.ctx, self.ws)

    def combine(self):
        self.M.moe_combine(self.ctx, self.w, self.ws, self.out)

    def forward(self):
        self.M.moe_forward(self.ctx, self.x, self.ids, self.w, self.ws, self.out)
        return self.out

    def status(self):
        return self.M.moe_read_device_status(self.ws)

    # decoded views
    def sf_bytes(self, name, rows):
        """UE8M0 bytes of the given rows, [len(rows), groups] (row indices in
        the a/h/y row space); MXFP8: [len(rows), 4 * groups], one byte per
        32-column block."""
        L, s = self.ctx.ws_layout, self.p
        groups = (s.K if name == "a_sf" else s.I) // 128
        sf = self.view(name).cpu().numpy()
        rows = np.asarray(rows, dtype=np.int64)
        if self.ctx.masked:
            e, pos = rows // s.max_m, rows % s.max_m
            bpe = (s.max_m + 127) // 128
            blk, r = e * bpe + pos // 128, pos % 128
        else:
            blk, r = rows // 128, rows % 128
        g = np.arange(groups)
        row_off = (16 * (r % 32) + 4 * (r // 32))[:, None]
        if self.ctx.mx:   # one chunk per group, the word's bytes its four 32-column blocks
            off = (blk[:, None] * groups + g[None, :]) * 512 + row_off
            return sf[(off[:, :, None] + np.arange(4)[None, None, :]).reshape(len(rows), 4 * groups)]
        # FP8 1x128: one chunk per four groups, group g in byte g % 4 of the word
        quads = -(-groups // 4)
        off = (blk[:, None] * quads + g[None, :] // 4) * 512 + row_off + g[None, :] % 4
        return sf[off]

    def decoded(self, name, rows):
        """fp64 values of rows of a or h as the GEMM consumes them."""
        v = self.view(name)
        rows_t = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=v.device)
        sel = v.index_select(0, rows_t).cpu()
        if not self.ctx.fp8:
            return bf16_to_f64(sel)
        q = oracle.e4m3_from_bits(sel.numpy())
        s = self.sf_bytes(name + "_sf", rows).astype(np.int64) - 127
        return oracle.dequant_groups(q, s, 32 if self.ctx.mx else 128)
