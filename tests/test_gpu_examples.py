"""Hand-worked examples (tests/golden) through the CUDA path."""
import numpy as np
import pytest

from tests import oracle_pins
from tests.gpu_parity import to_dev
from w4a16_compact_expert_gb300 import moe_w4a16

pytestmark = pytest.mark.gpu


def _run(experts, E, k, bias=None, flags=0, x_val=1.0):
    import torch
    m = moe_w4a16.MoELayer(256, 64, E, k, max_tokens=4)
    try:
        m.pack_experts(0, *experts)
        m.set_slot_table(np.arange(E))
        x = np.full((1, 256), x_val, np.float16)
        out, dbg = m.forward(to_dev(x), to_dev(np.zeros((E, 256), np.float16)), to_dev(bias), flags, debug=True)
        torch.cuda.synchronize()
        return out.float().cpu().numpy(), {k_: v.cpu().numpy() for k_, v in dbg.items()}
    finally:
        m.close()


def test_example_a_rounds_h_to_fp16():
    g = oracle_pins.load_golden("example_a.json")
    ex = oracle_pins.stack_experts(oracle_pins.example_expert(0x11, 0x11, 0x02))
    out, dbg = _run(ex, 1, 1)
    # the path rounds h to FP16 before the down projection: exactly 1497/2048
    assert np.all(out == g["expected_out_if_h_rounded_to_fp16"])
    assert dbg["ids"][0, 0] == 0 and dbg["weights"][0, 0] == 1.0


def test_example_b_sign_and_gate():
    g = oracle_pins.load_golden("example_b.json")
    ex = oracle_pins.stack_experts(oracle_pins.example_expert(0xFF, 0x11, 0x02))
    out, _ = _run(ex, 1, 1)
    h16 = float(np.float16(g["expected_out_every_h"]))
    assert np.all(out == h16)


def test_example_c_combine():
    g = oracle_pins.load_golden("example_c.json")
    ex = oracle_pins.stack_experts(oracle_pins.example_expert(0x11, 0x11, 0x02),
                                   oracle_pins.example_expert(0x11, 0x11, 0x0E))
    bias = np.array([0.0, np.log(3.0)], np.float32)
    out, dbg = _run(ex, 2, 2, bias=bias)
    assert dbg["ids"][0].tolist() == g["expected_ids"]
    assert np.allclose(dbg["weights"][0], g["expected_weights"], atol=1e-6)
    assert np.allclose(out, g["expected_out_every_h"], rtol=1e-3, atol=0)


def test_residual_prenorm_example():
    g = oracle_pins.load_golden("example_a.json")
    ex = oracle_pins.stack_experts(oracle_pins.example_expert(0x11, 0x11, 0x02))
    out, _ = _run(ex, 1, 1, flags=moe_w4a16.RESIDUAL | moe_w4a16.PRENORM, x_val=4.0)
    assert np.allclose(out, 4.0 + g["expected_out_every_h"], rtol=1e-3)
