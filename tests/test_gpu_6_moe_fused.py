"""The one-launch MoE (a few tokens) on the GPU against the CPU oracle.

One launch leaves its intermediates in the workspace (fp4_moe_workspace_layout
entries 15-21, slot order t * top_k + j), so the same staged parity as the
launch chain applies, each stage fed by the GPU's own previous stage:
  1 route              ids exact, weights 2e-6 relative
  2 dispatch-quantise  the dispatched hidden rows' codes / scale bytes bit-exact
  3 GEMM1 + SiLU*up    h within the bf16-rounding tolerance of the oracle's h
  4 requantise         s_gH = amax(GPU h of the expert) / 2688 (static: the
                       expert's scale) and the h codes / scale bytes bit-exact
                       against the oracle's quantiser on the GPU's h
  5 GEMM2 + combine    D and y within tolerance of the oracle's GEMM2 and
                       slot-order sum on the GPU's requantised h
and the output is the same bits on every run (the top-k sum has a fixed order).
"""
import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I
from util import bf16_to_np, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


class Fused:
    def __init__(self, F, O, T, E, k, H, Inter, seed, std, q=None, mw=None, static=None):
        self.T, self.E, self.k, self.H, self.I = T, E, k, H, Inter
        self.hidden = I.randn_bf16((T, H), seed + 1)
        self.logits = I.router_logits(T, E, seed + 2)
        if mw is None:
            w13 = I.expert_weights_bf16(E, 2 * Inter, H, seed + 3, std)
            w2 = I.expert_weights_bf16(E, H, Inter, seed + 4, std)
            mw = F.moe_prepack(w13.cuda(), w2.cuda())
            q = (O.quantize_experts(I.u16(w13)), O.quantize_experts(I.u16(w2)))
        self.mw, (self.q13, self.q2) = mw, q
        self.static = static
        kw = {} if static is None else dict(mode=1, static13=static[0], static2=static[1])
        self.ref = O.moe(I.u16(self.hidden), self.logits.numpy(), top_k=k, q13=self.q13, q2=self.q2, **kw)
        L = F.lib()
        self.ws = torch.zeros(L.fp4_moe_workspace_size(T, H, Inter, E, k), dtype=torch.uint8, device="cuda")
        self.off = F.moe_workspace_layout(T, H, Inter, E, k)
        assert len(self.off) >= 22
        self.hid_d, self.log_d = self.hidden.cuda(), self.logits.cuda()

    def view(self, entry, dtype, shape):
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        o = self.off[entry]
        return self.ws[o:o + nbytes].view(dtype).view(shape)

    def run(self, F, policy=None):
        st = self.static
        kw = {} if st is None else dict(mode=1, static13=st[0], static2=st[1])
        F.set_moe_policy(F.MOE_FUSED if policy is None else policy)
        try:
            out = F.moe(self.hid_d, self.log_d, self.mw, self.k, workspace=self.ws, **kw)
        finally:
            F.set_moe_policy(F.MOE_AUTO)
        torch.cuda.synchronize()
        F.device_status()
        return out


def fused_checks(F, O, c):
    T, E, k, H, Inter = c.T, c.E, c.k, c.H, c.I
    S = T * k
    r = c.ref
    out = c.run(F)
    y = bf16_to_np(out)
    # 1. route
    assert np.array_equal(c.view(0, torch.int32, (T, k)).cpu().numpy(), r["ids"])
    assert np.allclose(c.view(1, torch.float32, (T, k)).cpu().numpy(), r["weights"], rtol=2e-6, atol=0)
    order = r["order"]          # sorted position p -> slot t * k + j
    ids = r["ids"].ravel()      # expert of each slot
    # 2. dispatched hidden rows, slot order
    ac = c.view(20, torch.uint8, (S, H // 2)).cpu().numpy()
    asb = c.view(21, torch.uint8, (S, H // 16)).cpu().numpy()
    assert np.array_equal(ac[order], r["a_codes"])
    assert np.array_equal(asb[order], r["a_scales"])
    if c.static is None:
        assert np.float32(c.view(7, torch.float32, (E,))[0].item()) == np.float32(r["sgA"])
    # 3. h
    h_u16 = c.view(15, torch.int16, (S, Inter)).cpu().numpy().view(np.uint16)
    h = O.bf16_to_f32(h_u16).astype(np.float64)[order]
    G, Gm = r["G"], r["Gmag"]
    tau_g = 2.0 ** -18 * Gm + 2.0 ** -22 * np.abs(G)
    g, u = G[:, :Inter], G[:, Inter:]
    sg = O.silu(g)
    tau_h = 1.1 * np.abs(u) * tau_g[:, :Inter] + np.abs(sg) * tau_g[:, Inter:] + 2.0 ** -20 * np.abs(sg * u)
    check_close(h, r["h64"], np.zeros_like(h), floor=0.0, extra_tau=tau_h, what="h")
    # 4. requantisation of the GPU's h, per expert
    hc = c.view(16, torch.uint8, (S, Inter // 2)).cpu().numpy()
    hs = c.view(17, torch.uint8, (S, Inter // 16)).cpu().numpy()
    sgh_gpu = c.view(18, torch.float32, (E,)).cpu().numpy()
    c2, s2, g2 = c.q2
    D_ref = np.zeros((S, H))
    D_mag = np.zeros((S, H))
    for e in np.unique(ids):
        slots = np.nonzero(ids == e)[0]
        he = h_u16[slots]
        if c.static is None:
            sgh = O.nvfp4_global_scale(O.amax_bf16(he))
        else:
            sgh = np.float32(c.static[1][e])
        assert np.float32(sgh_gpu[e]) == np.float32(sgh), (e, sgh_gpu[e], sgh)
        want_c, want_s = O.quantize_nvfp4_given_scale(he, sgh)
        assert np.array_equal(hc[slots], want_c), "requantised h codes of expert %d" % e
        assert np.array_equal(hs[slots], want_s), "requantised h scale bytes of expert %d" % e
        D_ref[slots], D_mag[slots] = O.gemm(O.NVFP4, want_c, want_s, sgh, c2[e], s2[e], g2[e])
    # 5. D and the slot-order combine (fp32: k roundings of the sum on top)
    D = c.view(19, torch.float32, (S, H)).cpu().numpy().astype(np.float64)
    tau_d = 2.0 ** -18 * D_mag + 2.0 ** -22 * np.abs(D_ref)
    assert np.all(np.abs(D - D_ref) <= tau_d + 1e-30), "D"
    w = r["weights"].ravel()
    y_ref = np.zeros((T, H))
    y_mag = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            y_ref[t] += w[t * k + j] * D_ref[t * k + j]
            y_mag[t] += abs(w[t * k + j]) * D_mag[t * k + j]
    check_close(y, y_ref, y_mag, what="y", extra_tau=k * 2.0 ** -23 * y_mag)
    # end to end against the oracle's own chain (norm-wise; requant flips allowed)
    err = np.linalg.norm(y - r["y"]) / np.linalg.norm(r["y"])
    assert err <= 3e-3, err
    # the same bits on a second run
    y2 = bf16_to_np(c.run(F))
    assert np.array_equal(y, y2)
    return y


@pytest.mark.parametrize("T,E,k,H,Inter", [(1, 8, 2, 256, 256), (5, 8, 2, 512, 256), (16, 16, 4, 256, 512),
                                           (3, 64, 8, 512, 768), (16, 128, 8, 256, 256)])
def test_moe_fused_small(F, O, T, E, k, H, Inter):
    c = Fused(F, O, T, E, k, H, Inter, seed=70 + T, std=0.1)
    fused_checks(F, O, c)


@pytest.mark.parametrize("T", [1, 16])
def test_moe_fused_static(F, O, T):
    E = 16
    rng = np.random.default_rng(T)
    st = ((rng.permutation(np.linspace(3.5, 6.0, E)) / 2688).astype(np.float32),
          (rng.permutation(np.linspace(1.5, 5.0, E)) / 2688).astype(np.float32))
    c = Fused(F, O, T, E, 4, 512, 256, seed=90 + T, std=0.1, static=st)
    fused_checks(F, O, c)


def test_moe_fused_matches_chain(F, O):
    """The one-launch MoE and the launch chain agree within the tolerance."""
    c = Fused(F, O, 12, 32, 4, 512, 256, seed=5, std=0.1)
    y_fused = bf16_to_np(c.run(F))
    y_chain = bf16_to_np(c.run(F, F.MOE_CHAIN))
    assert np.linalg.norm(y_fused - y_chain) / np.linalg.norm(y_chain) <= 3e-3


@pytest.fixture(scope="module")
def full_experts(F, O):
    E, H, Inter = 128, 2048, 768
    w13 = I.expert_weights_bf16(E, 2 * Inter, H, 103)
    w2 = I.expert_weights_bf16(E, H, Inter, 104)
    mw = F.moe_prepack(w13.cuda(), w2.cuda())
    return mw, (O.quantize_experts(I.u16(w13)), O.quantize_experts(I.u16(w2)))


@pytest.mark.parametrize("T", [1, 8, 16])
def test_moe_fused_full_size(F, O, full_experts, T):
    """128 experts, top-8, hidden 2048, intermediate 768, in one launch."""
    mw, q = full_experts
    c = Fused(F, O, T, 128, 8, 2048, 768, seed=3, std=0.02, q=q, mw=mw)
    fused_checks(F, O, c)


def test_moe_fused_full_size_static(F, O, full_experts):
    mw, q = full_experts
    rng = np.random.default_rng(7)
    st = ((rng.permutation(np.linspace(3.5, 6.0, 128)) / 2688).astype(np.float32),
          (rng.permutation(np.linspace(1.5, 5.0, 128)) / 2688).astype(np.float32))
    c = Fused(F, O, 4, 128, 8, 2048, 768, seed=11, std=0.02, q=q, mw=mw, static=st)
    fused_checks(F, O, c)
