"""The two MoE expert kernels of the decode step, called through the C ABI
(hy_op_moe_gateup: top-k of the router logits in every CTA, then the picked
experts' and the shared expert's gate/up rows with SwiGLU; hy_op_moe_down:
the weighted down projections added to the residual), against the FP64
oracle: expert ids bit-exact (the logits are drawn with a clear top-k gap),
routing weights, and every output element within its FP32 bound."""
import numpy as np
import pytest

from oracle import oracle as orc
from synth import gen
from tests.gpu_util import bf16_tensor, gamma, to_np

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build, capi
    build.build()
    return capi.lib()


def wide(b):
    return gen.bf16_bits_to_f32(b).astype(np.float64)


@pytest.mark.parametrize("E,K,Fe,H", [(16, 4, 64, 256), (256, 8, 512, 2048), (511, 16, 64, 512)])
def test_moe_gateup_and_down(L, E, K, Fe, H):
    import torch
    rng = np.random.default_rng(E + K + Fe)
    def mats(*shape):
        return gen.f32_to_bf16_bits((rng.standard_normal(shape) * 0.02).astype(np.float32))
    eg, eu, ed = mats(E, Fe, H), mats(E, Fe, H), mats(E, H, Fe)
    sg, su, sd = mats(Fe, H), mats(Fe, H), mats(H, Fe)
    # router logits with a gap of at least 0.01 between neighbours in rank order
    order = rng.permutation(E)
    logits = np.zeros(E + 1, dtype=np.float32)
    logits[order] = np.linspace(2.0, -2.0, E).astype(np.float32) + rng.uniform(0, 0.002, E).astype(np.float32)
    logits[E] = np.float32(rng.standard_normal())
    x = rng.standard_normal(H).astype(np.float32)
    g = rng.uniform(0.5, 1.5, H).astype(np.float32)
    y0 = rng.standard_normal(H).astype(np.float32)
    dev = [bf16_tensor(a) for a in (eg, eu, ed, sg, su, sd)]
    ld, xd, gd = (torch.from_numpy(a).cuda() for a in (logits, x, g))
    h = torch.empty((K + 1) * Fe, dtype=torch.float32, device="cuda")
    ids = torch.empty(K, dtype=torch.int32, device="cuda")
    w = torch.empty(K + 1, dtype=torch.float32, device="cuda")
    y = torch.from_numpy(y0.copy()).cuda()
    st = torch.cuda.current_stream().cuda_stream
    assert L.hy_op_moe_gateup(dev[0].data_ptr(), dev[1].data_ptr(), dev[3].data_ptr(), dev[4].data_ptr(), E, K, Fe, H,
                              ld.data_ptr(), xd.data_ptr(), gd.data_ptr(), 1e-6, h.data_ptr(), ids.data_ptr(),
                              w.data_ptr(), st) == 0, L.hy_last_error()
    assert L.hy_op_moe_down(dev[2].data_ptr(), dev[5].data_ptr(), E, K, Fe, H, ids.data_ptr(), w.data_ptr(),
                            h.data_ptr(), y.data_ptr(), st) == 0, L.hy_last_error()
    torch.cuda.synchronize()
    # routing: ids in selection order, weights = softmax of the picked logits, shared gate = sigmoid
    want_ids = orc.topk(logits[:E].astype(np.float64), K)
    np.testing.assert_array_equal(to_np(ids), want_ids)
    want_w = np.r_[orc.softmax(logits[want_ids].astype(np.float64)), orc.lib().orc_sigmoid(float(logits[E]))]
    np.testing.assert_allclose(to_np(w), want_w, rtol=1e-5, atol=1e-7)
    # gate/up + SwiGLU per slot
    xh = orc.rmsnorm(x, g, 1e-6)
    rows_g = [wide(eg[e]) for e in want_ids] + [wide(sg)]
    rows_u = [wide(eu[e]) for e in want_ids] + [wide(su)]
    a = np.concatenate([r @ xh for r in rows_g])
    u = np.concatenate([r @ xh for r in rows_u])
    sa = np.concatenate([np.abs(r) @ np.abs(xh) for r in rows_g])
    su_ = np.concatenate([np.abs(r) @ np.abs(xh) for r in rows_u])
    ref_h = a / (1 + np.exp(-a)) * u
    rel = gamma(H + 64) + 16 * U32
    tol_h = 1.1 * rel * sa * np.abs(u) + rel * su_ * np.abs(a) + 64 * U32 * np.abs(ref_h) + 1e-30
    gh = to_np(h)
    assert np.all(np.abs(gh - ref_h) <= tol_h), f"h: worst {(np.abs(gh - ref_h) / tol_h).max():.3g}"
    # down: y = y0 + sum_s w_s Wd_s h_s, computed from the kernel's own h and w (the step's inputs)
    wv = to_np(w).astype(np.float64)
    downs = [wide(ed[e]) for e in want_ids] + [wide(sd)]
    ref_y = y0.astype(np.float64).copy()
    abs_y = np.abs(y0).astype(np.float64)
    for s_, D in enumerate(downs):
        hs = gh[s_ * Fe:(s_ + 1) * Fe].astype(np.float64) * wv[s_]
        ref_y += D @ hs
        abs_y += np.abs(D) @ np.abs(hs)
    tol_y = (gamma((K + 1) * Fe + 64) + 16 * U32) * abs_y + 1e-30
    gy = to_np(y)
    assert np.all(np.abs(gy - ref_y) <= tol_y), f"y: worst {(np.abs(gy - ref_y) / tol_y).max():.3g}"
