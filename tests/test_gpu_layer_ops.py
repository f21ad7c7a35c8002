"""GPU parity of the GDN causal convolution with ring rollback and of the gated
RMSNorm + E4M3 quantisation (libgdnreplay, through the C ABI of include/gdnlayer.h)
against the CPU oracle on the same seeded inputs.

Tolerances, derived from the arithmetic (fp32 on the GPU, fp64 in the oracle):
* convolution, fp32 y: each output is bias + W <= 4 fused multiply-adds and a SiLU
  (__expf and __fdividef, relative error about 2^-21 each), so |d| <= 2^-20 S + 1e-7
  with S = |bias| + sum_j |w_j x_j| per element;
* convolution, bf16 y: the bf16 rounding of that fp32 value: exact wherever the fp64
  value is farther than that bound from a rounding midpoint, else either neighbour;
* norm codes: every factor is a product (no cancellation), so the fp32 value is within
  1e-5 relative of the fp64 one; codes exact outside that band around an E4M3
  midpoint, either neighbour inside it;
* ring contents and write positions (copies and integer updates): bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from harness import assert_bf16_rounding, assert_e4m3_codes
from synth.layer_ops import CONV_WORKLOADS, NORM_WORKLOADS, conv_block, initial_conv_layer, norm_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def _dims(wl):
    import speculative_decode_recurrent_gb300 as lib
    dt = {"bf16": lib.DTYPE_BF16, "fp32": lib.DTYPE_F32}
    return lib.ConvDims(B=wl.B, D=wl.D, W=wl.W, T=wl.T, cap=wl.cap, n_slot=wl.n_slot, act=wl.act,
                        in_dtype=dt[wl.in_dtype], out_dtype=dt[wl.out_dtype])


class ConvPair:
    def __init__(self, wl, layer=0):
        import speculative_decode_recurrent_gb300 as lib
        self.wl = wl
        init = initial_conv_layer(wl, layer)
        self.init = init
        self.gpu = lib.ConvLayer(_dims(wl), init)
        self.orc = oracle.ConvLayer(oracle.ConvDims(B=wl.B, D=wl.D, W=wl.W, T=wl.T, cap=wl.cap,
                                                    n_slot=wl.n_slot, act=wl.act), init)
        self.layer = layer

    def band(self, x):
        """Per-element bound S of the fp32 arithmetic (see the module docstring)."""
        wl, o = self.wl, self.orc
        xs = x.double().numpy()
        S = np.zeros((wl.B, wl.T, wl.D))
        for b in range(wl.B):
            s = o.state_idx[b]
            win = [o.ring[s, (o.pos[s] - (wl.W - 1) + j) % wl.cap] for j in range(wl.W - 1)]
            seq = np.concatenate([np.array(win).reshape(wl.W - 1, wl.D), xs[b]], 0)
            for t in range(wl.T):
                S[b, t] = np.abs(o.bias) + sum(np.abs(o.w[:, j] * seq[t + j]) for j in range(wl.W))
        return 2.0 ** -20 * S + 1e-7

    def step(self, s, accepted=None):
        wl = self.wl
        blk = conv_block(wl, self.layer, s)
        acc = blk["accepted"] if accepted is None else torch.as_tensor(accepted, dtype=torch.int32)
        band = self.band(blk["x"])
        y = torch.empty(wl.B, wl.T, wl.D, dtype=wl.torch_dtype("out_dtype"), device="cuda")
        self.gpu.verify(blk["x"].cuda(), y)
        y_ref = self.orc.verify(blk["x"])
        self.gpu.accept(acc.cuda())
        self.orc.accept(acc.numpy())
        torch.cuda.synchronize()
        tag = f"{wl.name}/step{s}"
        amb = 0
        if wl.out_dtype == "fp32":
            err = np.abs(y.cpu().double().numpy() - y_ref)
            assert (err <= band).all(), f"{tag}: max excess {float((err - band).max()):.3e}"
        else:
            amb = assert_bf16_rounding(f"y {tag}", y, y_ref, band)
        t = self.gpu.t
        np.testing.assert_array_equal(t["pos"].cpu().numpy(), self.orc.pos, err_msg=tag)
        np.testing.assert_array_equal(t["ring"].cpu().double().numpy(), self.orc.ring, err_msg=tag)
        assert int(self.gpu.status.item()) == int(self.orc.status[0]) == 0, tag
        return amb


@pytest.mark.parametrize("name,steps", [("conv_decode", 12), ("conv_edge", 20), ("conv_w3_f32", 30),
                                        ("conv_w2_bf16", 30), ("conv_w1", 10)])
def test_conv_parity_multistep(name, steps):
    """verify -> accept over many steps (the ring wraps; forced accepts 0..16 on the
    tightest ring): outputs, ring bytes and write positions against the oracle."""
    pr = ConvPair(CONV_WORKLOADS[name])
    amb = sum(pr.step(s) for s in range(steps))
    wl = pr.wl
    assert amb <= 0.02 * steps * wl.B * wl.T * wl.D      # the band is not so wide that it decides nothing


def test_conv_full_rejection_is_bit_identical():
    """Accepting nothing leaves the write positions, and the next verify of the same
    draft gives the same outputs bit for bit."""
    wl = CONV_WORKLOADS["conv_decode"]
    pr = ConvPair(wl)
    blk = conv_block(wl, 0, 0)
    x = blk["x"].cuda()
    y1 = torch.empty(wl.B, wl.T, wl.D, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    pos0 = pr.gpu.t["pos"].clone()
    pr.gpu.verify(x, y1)
    pr.gpu.accept(torch.zeros(wl.B, dtype=torch.int32, device="cuda"))
    pr.gpu.verify(x, y2)
    torch.cuda.synchronize()
    assert torch.equal(pr.gpu.t["pos"], pos0)
    assert torch.equal(y1, y2)


def test_conv_status_bits_and_guard_bands():
    """A bad slot, a corrupt write position and bad accepted counts are reported in the
    status word and skip the sequence; nothing is written past any tensor's end."""
    import speculative_decode_recurrent_gb300 as lib
    wl = CONV_WORKLOADS["conv_w3_f32"]
    init = initial_conv_layer(wl, 0)
    d = _dims(wl)
    pad = 4096

    def padded(t, fill):
        flat = torch.full((t.numel() + pad,), fill, dtype=t.dtype, device="cuda")
        flat[:t.numel()] = t.reshape(-1).cuda()
        return flat, flat[:t.numel()].view(t.shape)

    ring_f, ring = padded(init["ring"], float("nan"))
    pos_f, pos = padded(init["pos"], -7)
    idx = init["state_idx"].clone().cuda()
    blk = conv_block(wl, 0, 0)
    y_f, y = padded(torch.zeros(wl.B, wl.T, wl.D), float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w, b = init["weight"].cuda(), init["bias"].cuda()
    lib.gdn_conv_verify(d, ring, pos, idx, blk["x"].cuda(), w, b, y, st)
    lib.gdn_conv_accept(d, pos, idx, blk["accepted"].cuda(), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for f, t in ((ring_f, ring), (y_f, y)):
        assert torch.isnan(f[t.numel():]).all()
    assert (pos_f[pos.numel():] == -7).all()
    # a slot out of range, a corrupt position, bad accepted counts
    idx[0] = wl.n_slot + 3
    pos[idx[1].long()] = wl.cap
    y.fill_(5.0)
    lib.gdn_conv_verify(d, ring, pos, idx, blk["x"].cuda(), w, b, y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == lib.STATUS_BAD_SLOT | lib.STATUS_BAD_LEN
    assert bool((y[0] == 5.0).all()) and bool((y[1] == 5.0).all()) and not bool((y[2] == 5.0).all())
    st.zero_()
    p0 = pos.clone()
    lib.gdn_conv_accept(d, pos, init["state_idx"].cuda(),
                        torch.tensor([-1, 0, wl.T + 1, 0, 0], dtype=torch.int32, device="cuda"), st)
    torch.cuda.synchronize()
    assert int(st.item()) & lib.STATUS_BAD_ACCEPT
    sl = init["state_idx"].long()
    assert int(pos[sl[0]]) == int(p0[sl[0]]) and int(pos[sl[2]]) == int(p0[sl[2]])


# --------------------------------------------------------- gated RMSNorm + E4M3
def _norm_run(o, z, w, eps, inv_scale):
    import speculative_decode_recurrent_gb300 as lib
    q = torch.empty(o.shape, dtype=torch.uint8, device="cuda")
    lib.gdn_gated_rmsnorm_fp8(o.cuda(), z.cuda(), w.cuda(), eps, inv_scale, q)
    torch.cuda.synchronize()
    return q.cpu().numpy()


@pytest.mark.parametrize("name", sorted(NORM_WORKLOADS))
def test_norm_fp8_codes(name):
    wl = NORM_WORKLOADS[name]
    inp = norm_inputs(wl)
    q = _norm_run(inp["o"], inp["z"], inp["weight"], wl.eps, wl.inv_scale)
    ref_q, ref_v = oracle.gated_rmsnorm_fp8(inp["o"].double().numpy(), inp["z"].double().numpy(),
                                            inp["weight"].double().numpy(), wl.eps, wl.inv_scale)
    amb = assert_e4m3_codes(name, q, ref_q, ref_v, 1e-5)
    assert amb <= 0.01 * q.size
    # the workload reaches saturation, subnormals and both signs
    assert ((ref_q & 0x7F) == 0x7E).any() and ((ref_q & 0x78) == 0).any() and (ref_q & 0x80).any()


def test_norm_fp8_on_verify_outputs():
    """The norm on the GDN outputs of a decode24 layer-step (the oracle's verify outputs,
    rounded to fp32, feed both sides), gated by a bf16 z."""
    import synth
    from harness import oracle_dims
    wl = synth.WORKLOADS["decode24"]
    init = synth.initial_layer(wl, 0, B=8)
    orc = oracle.Layer(oracle_dims(wl, B=8), init)
    o_ref = orc.verify(synth.draft_block(wl, 0, 0, B=8))
    o = torch.from_numpy(o_ref).float().reshape(-1, wl.dv).contiguous()
    g = torch.Generator().manual_seed(99)
    z = (2.0 * torch.randn(o.shape, generator=g)).bfloat16().contiguous()
    w = (1 + 0.1 * torch.randn(wl.dv, generator=g)).float()
    q = _norm_run(o, z, w, 1e-6, 50.0)
    ref_q, ref_v = oracle.gated_rmsnorm_fp8(o.double().numpy(), z.double().numpy(), w.double().numpy(),
                                            1e-6, 50.0)
    amb = assert_e4m3_codes("verify outputs", q, ref_q, ref_v, 1e-5)
    assert amb <= 0.01 * q.size
