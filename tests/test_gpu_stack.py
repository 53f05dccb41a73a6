"""The 16-layer OLMoE-shaped stack, x <- x + MoE(x / rms(x)), against the
oracle layer by layer with teacher forcing.

Each GPU layer l runs on the GPU's own FP16 x_l; the oracle's layer l takes
the same x_l, and every layer output is held to the acceptance bars of a
single layer (ids bit-exact on tokens that are not near ties, normwise
relative error <= 2e-3, max error <= 1e-2 max|ref|).  Because the residual
dominates deep layers, the MoE term alone (flag PRENORM without RESIDUAL) is
checked the same way at every layer.  The error of the whole one-token chain
against the oracle's own chain (float64 end to end) is printed, not gated.

The weights are drawn on the host (synth.olmoe_stack), so the oracle sees
exactly what the GPU does.  Token sets: T = 1 and 8 (single-launch decode
kernel), T = 64 (separate-launch decode kernels) and T = 64 forced onto the
grouped GEMM.  The oracle treats tokens independently, so one oracle call
per layer covers all sets; the 16 layers' calls run on a thread pool (numpy
releases the interpreter lock in its array kernels).

The stacked-layer reading (pre-norm with residual) is the one the library
takes for deep stacks: the literal x <- x + MoE(x) leaves FP16 range within
a few layers with these weight distributions.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as F, synth

pytestmark = pytest.mark.gpu

SETS = [(1, 0), (8, 0), (64, 0), (64, F.FORCE_GEMM)]
NL = 16


def test_stack_teacher_forced():
    import torch
    layers = synth.olmoe_stack(NL)
    H = synth.OLMOE.hidden
    k = synth.OLMOE.top_k
    x0 = [synth.draw_x(synth.SEED_OLMOE_STACK, T, H) for T, _ in SETS]
    m = gp.make_handle(layers[0], 64)
    xs = [list(x0)]            # xs[l][set]: GPU FP16 input of layer l
    outs, moes, dbgs = [], [], []
    try:
        for li, layer in enumerate(layers):
            if li:
                m.pack_experts(0, *layer.experts.arrays())   # identity slot table
            nxt, mo, db = [], [], []
            for (T, force), x in zip(SETS, xs[li]):
                out, dbg = gp.gpu_forward(m, layer, x, F.RESIDUAL | F.PRENORM | force)
                moe, _ = gp.gpu_forward(m, layer, x, F.PRENORM | force)
                nxt.append(out.astype(np.float16))
                mo.append(moe)
                db.append(dbg)
            assert m.get_status() == (F.OK, 0), li
            assert all(np.isfinite(o).all() for o in nxt), li
            outs.append([o.astype(np.float64) for o in nxt])
            moes.append(mo)
            dbgs.append(db)
            xs.append(nxt)
        torch.cuda.synchronize()
    finally:
        m.close()

    sizes = [T for T, _ in SETS]
    cut = np.cumsum([0] + sizes)

    def teacher_forced(li):
        xin = np.concatenate(xs[li])
        return moe_oracle.moe_layer(xin, layers[li].router_w, layers[li].bias, layers[li].experts.arrays(),
                                    k, moe_oracle.FLAG_RESIDUAL | moe_oracle.FLAG_PRENORM)

    def own_chain():
        # the oracle's chain from x_0 of the one-token set in float64 (no FP16
        # rounding between layers; one token keeps the 16 sequential calls short)
        x = x0[0].astype(np.float64)
        for layer in layers:
            x = moe_oracle.moe_layer(x, layer.router_w, layer.bias, layer.experts.arrays(), k,
                                     moe_oracle.FLAG_RESIDUAL | moe_oracle.FLAG_PRENORM).out
        return x

    with ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as ex:
        chain = ex.submit(own_chain)
        refs = list(ex.map(teacher_forced, range(NL)))
        x_end = chain.result()

    worst = 0.0
    for li in range(NL):
        ref = refs[li]
        assert not ref.overflow.any(), li
        for si, (T, force) in enumerate(SETS):
            sl = slice(cut[si], cut[si + 1])
            flagged = ref.near_tie[sl]
            gp.assert_routing(dbgs[li][si], ref.ids[sl], ref.weights[sl], flagged, synth.OLMOE.num_experts)
            keep = ~flagged
            worst = max(worst, gp.assert_output(outs[li][si], ref.out[sl], keep))
            moe_ref = ref.out[sl] - np.concatenate(xs[li])[sl].astype(np.float64)
            gp.assert_output(moes[li][si], moe_ref, keep)
    d = outs[-1][0] - x_end
    print(f"stack T=1: end-to-end rel err after {NL} layers {np.linalg.norm(d) / np.linalg.norm(x_end):.2e} "
          f"(not gated); rms(x_16) {np.sqrt(np.mean(x_end ** 2)):.1f}")
    print(f"worst per-layer rel err {worst:.2e}")
