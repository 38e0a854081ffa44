"""Device-side layers for the GPU parity tests: weights generated on the
device by the seeded generator and packed by the library, with the matching
oracle-side rows regenerated on the host (the oracle never sees device data)."""
import numpy as np
import torch

import oracle
import synth


class DevLayer:
    """One layer's weights generated on the device and packed by the library."""

    def __init__(self, mt, wl, layer):
        self.wl, self.l = wl, layer
        d, f, g = wl.d, wl.f, wl.group
        sd = lambda t: synth.seed_for(wl.wid, layer, t)
        self.sd = sd
        bf = torch.bfloat16
        self.w = torch.empty(d, dtype=bf, device="cuda")
        synth.device_bf16(self.w, sd(synth.T_NORM_W), synth.NORM_W)
        if wl.fmt == synth.FMT_BF16:
            self.Wg = torch.empty(f, d, dtype=bf, device="cuda")
            self.Wu = torch.empty(f, d, dtype=bf, device="cuda")
            self.Wd = torch.empty(d, f, dtype=bf, device="cuda")
            for W, t in ((self.Wg, synth.T_WG), (self.Wu, synth.T_WU), (self.Wd, synth.T_WD)):
                synth.device_bf16(W, sd(t), wl.weight_dist)
            self.sgu = self.bgu = self.sdn = self.bdn = None
        else:
            b = wl.bits
            mx = synth.is_mx(wl.fmt)
            sdt = torch.uint8 if mx else bf
            self.Wg = torch.empty(f, d * b // 8, dtype=torch.uint8, device="cuda")
            self.Wu = torch.empty_like(self.Wg)
            self.Wd = torch.empty(d, f * b // 8, dtype=torch.uint8, device="cuda")
            self.sgu = torch.empty(2, f, d // g, dtype=sdt, device="cuda")
            self.sdn = torch.empty(d, f // g, dtype=sdt, device="cuda")
            self.bgu = None if mx else torch.empty_like(self.sgu)
            self.bdn = None if mx else torch.empty_like(self.sdn)
            tmp = torch.empty(d * f, dtype=torch.float32, device="cuda")
            for (dst, s_, b_, N, K, t) in ((self.Wg, self.sgu[0], None if mx else self.bgu[0], f, d, synth.T_WG),
                                           (self.Wu, self.sgu[1], None if mx else self.bgu[1], f, d, synth.T_WU),
                                           (self.Wd, self.sdn, self.bdn, d, f, synth.T_WD)):
                W32 = tmp[:N * K].view(N, K)
                synth.device_f32(W32, sd(t), wl.weight_dist)
                if mx:
                    mt.mt_pack_mx(W32, N, K, b, dst, s_)
                else:
                    mt.mt_pack_affine(W32, N, K, g, b, dst, s_, b_)
            del tmp
        torch.cuda.synchronize()

    def oracle_rows(self, tensor, rows, N, K):
        """Oracle-side weight rows [rows] of matrix `tensor` ([N][K])."""
        wl = self.wl
        W32 = np.stack([synth.host_f32(K, self.sd(tensor), wl.weight_dist, offset=int(n) * K) for n in rows])
        if synth.is_mx(wl.fmt):
            return oracle.Weight.from_f32_mx(W32, wl.bits)
        return oracle.Weight.from_f32(W32, wl.bits, wl.group)


def run_layer(mt, L, v, r, M):
    wl = L.wl
    d, f = wl.d, wl.f
    out_sum = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    out_norm = torch.empty_like(out_sum)
    h = torch.empty(M, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(M, d, dtype=torch.bfloat16, device="cuda")
    mt.mt_add_rmsnorm(v, r, L.w, wl.eps, out_sum, out_norm)
    mt.mt_swiglu_gateup(out_norm, L.Wg, L.Wu, L.sgu, L.bgu, wl.group, h, fmt=wl.fmt)
    mt.mt_down_residual(h, L.Wd, L.sdn, L.bdn, wl.group, out_sum, y, fmt=wl.fmt)
    torch.cuda.synchronize()
    return out_sum, out_norm, h, y


def host_acts(wl, layer, M):
    sd = lambda t: synth.seed_for(wl.wid, layer, t)
    v = synth.host_bf16(M * wl.d, sd(synth.T_VALUES), synth.ACT).reshape(M, wl.d)
    r = synth.host_bf16(M * wl.d, synth.seed_for(wl.wid, 0, synth.T_RESIDUAL), synth.ACT).reshape(M, wl.d)
    w = synth.host_bf16(wl.d, sd(synth.T_NORM_W), synth.NORM_W)
    return v, r, w


def full_oracle_layer(L, v, r, w):
    wl = L.wl
    d, f = wl.d, wl.f
    Wg = L.oracle_rows(synth.T_WG, range(f), f, d)
    Wu = L.oracle_rows(synth.T_WU, range(f), f, d)
    Wd = L.oracle_rows(synth.T_WD, range(d), d, f)
    return oracle.mlp_layer(v, r, w, wl.eps, Wg, Wu, Wd), (Wg, Wu, Wd)


def plan_layer(L):
    """The layer as an ``mt_mlp_layer`` mapping for mt_mlp_plan_create."""
    return dict(norm_weight=L.w, Wg=L.Wg, Wu=L.Wu, gu_scales=L.sgu, gu_biases=L.bgu, Wd=L.Wd,
                d_scales=L.sdn, d_biases=L.bdn)


class DevProj:
    """One projection's weight (and bias) generated on the device and packed by
    the library, with oracle-side rows regenerated on the host."""

    def __init__(self, mt, wl, p, layer=0):
        self.wl, self.p, self.l = wl, p, layer
        sd = lambda t: synth.seed_for(wl.wid, layer, t)
        self.sd = sd
        N, K, g = p.N, p.K, wl.group
        bf = torch.bfloat16
        if wl.fmt == synth.FMT_BF16:
            self.W = torch.empty(N, K, dtype=bf, device="cuda")
            synth.device_bf16(self.W, sd(p.tensor), wl.weight_dist)
            self.s = self.b = None
        else:
            self.W = torch.empty(N, K * wl.bits // 8, dtype=torch.uint8, device="cuda")
            self.s = torch.empty(N, K // g, dtype=bf, device="cuda")
            self.b = torch.empty_like(self.s)
            tmp = torch.empty(N, K, dtype=torch.float32, device="cuda")
            synth.device_f32(tmp, sd(p.tensor), wl.weight_dist)
            mt.mt_pack_affine(tmp, N, K, g, wl.bits, self.W, self.s, self.b)
            del tmp
        self.bias = None
        if p.bias is not None:
            self.bias = torch.empty(N, dtype=bf, device="cuda")
            synth.device_bf16(self.bias, sd(p.bias), synth.PROJ_BIAS)
        torch.cuda.synchronize()

    def run(self, mt, x, out):
        mt.mt_linear_bias(x, self.W, self.s, self.b, self.wl.group, self.bias, out, fmt=self.wl.fmt)

    def oracle_rows(self, rows):
        """Oracle-side weight rows and bias entries for output columns `rows`."""
        wl, p = self.wl, self.p
        K = p.K
        if wl.fmt == synth.FMT_BF16:
            W = np.stack([synth.host_bf16(K, self.sd(p.tensor), wl.weight_dist, offset=int(n) * K)
                          for n in rows])
            Wo = oracle.Weight(oracle.FMT_BF16, W)
        else:
            W32 = np.stack([synth.host_f32(K, self.sd(p.tensor), wl.weight_dist, offset=int(n) * K)
                            for n in rows])
            Wo = oracle.Weight.from_f32(W32, wl.bits, wl.group)
        bias = None
        if p.bias is not None:
            full = synth.host_bf16(p.N, self.sd(p.bias), synth.PROJ_BIAS)
            bias = full[np.asarray(list(rows), dtype=np.int64)]
        return Wo, bias
