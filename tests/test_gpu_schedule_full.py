"""The DelayedScaling schedule at the CodonFM-5B sizes (M = 15872 tokens, hidden 4096,
intermediate 16384), and the recipe state's checkpoint.

1. Two full-size layers (eight linears) with Student-t(3) activations carrying 0.1 % outliers
   x100, run for enough steps that the 16-slot histories wrap (and with the 1024-slot
   history of the NeMo configuration).  Each step multiplies every tensor by its own power of
   two (exact in bf16), so amaxes move and delayed scales saturate.  The oracle takes the amax
   of each full-size tensor once; a power-of-two scaling multiplies it exactly, so the oracle's
   amax at each step is that amax times the step's power of two.  Histories, scales and
   scale_invs bit-exact after every step.
   ("Introduction to FP8 training using Transformer Engine": DelayedScaling with
   amax_history_len 16, algo max, HYBRID formats; NeMo key fp8_amax_history_len 1024.)
2. Save / restore: the FP8 metadata a module keeps beside its weights (its "_extra_state" in
   the pages' HuggingFace BERT example) is the recipe state; a run restored from a mid-run
   checkpoint continues bit-identically.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_transformer_gb300.linear import ScheduleStep
from oracle import quantize as Q
from oracle import recipes as Rc
from synthetic import gaussian, seed_for, student_t_outliers
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

M, H, F = 15872, 4096, 16384
SHAPES = [(H, 3 * H), (H, H), (H, F), (F, H)]


def _layers(n_layers, m=M, shapes=SHAPES):
    out = []
    for l in range(n_layers):
        lin = []
        for i, (k_in, n_out) in enumerate(shapes):
            s = seed_for(5, 100 * l + i, 0)
            lin.append((student_t_outliers((m, k_in), s, device=G.DEV),
                        gaussian((n_out, k_in), 0.02, s + 1, device=G.DEV),
                        gaussian((m, n_out), 1e-3, s + 2, device=G.DEV),
                        gaussian((n_out,), 0.02, s + 3, dtype=torch.float32, device=G.DEV)))
        out.append(lin)
    return out


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("L", [16, 1024])
def test_full_size_schedule_histories_and_scales(L):
    layers = _layers(2)
    sched = ScheduleStep(layers, history_len=L)
    tensors = [t for lin in layers for (x, w, dy, _) in lin for t in (x, w, dy)]
    base_amax = [Q.amax(G.f32_np(t)) for t in tensors]            # the oracle's whole-tensor amaxes
    n_lin = len(tensors) // 3
    ox = [Rc.DelayedScalingState("e4m3", L) for _ in range(2 * n_lin)]
    od = [Rc.DelayedScalingState("e5m2", L) for _ in range(n_lin)]
    rng = np.random.default_rng(L)
    expo = np.zeros(len(tensors), np.int64)
    steps = 2 * 16 + 3
    for t in range(steps):
        k = np.clip(expo + rng.integers(-2, 3, size=len(tensors)), -6, 6) - expo   # |2^expo| stays in 2^-6..2^6
        for tt, kk in zip(tensors, k):
            tt.mul_(2.0 ** int(kk))                                # exact in bf16
        expo += k
        sched.run(t)
        for i in range(n_lin):
            a = [np.float32(base_amax[3 * i + j] * np.float32(2.0 ** int(expo[3 * i + j]))) for j in range(3)]
            ox[2 * i].update(a[0], t)
            ox[2 * i + 1].update(a[1], t)
            od[i].update(a[2], t)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(sched.fwd.amax),
                                      np.array([base_amax[3 * i + j] * np.float32(2.0 ** int(expo[3 * i + j]))
                                                for i in range(n_lin) for j in (0, 1)], np.float32).view(np.uint32))
        for dev_state, states in ((sched.fwd, ox), (sched.bwd, od)):
            np.testing.assert_array_equal(_bits(dev_state.scale), np.array([s.scale for s in states], np.float32).view(np.uint32))
            np.testing.assert_array_equal(_bits(dev_state.scale_inv),
                                          np.array([s.scale_inv for s in states], np.float32).view(np.uint32))
            np.testing.assert_array_equal(_bits(dev_state.hist).reshape(-1, L), np.stack([s.hist for s in states]).view(np.uint32))
    assert any(s.scale != 1.0 for s in ox) and any(s.scale != 1.0 for s in od)
    G.check_no_device_error()


def test_recipe_state_checkpoint_restores_bit_identically():
    shapes = [(256, 768), (256, 256), (256, 1024), (1024, 256)]
    L, steps, cut = 16, 30, 11

    def perturb(layers, t):
        r = np.random.default_rng(t)
        for lin in layers:
            for x, w, dy, _ in lin:
                for tt in (x, w, dy):
                    tt.mul_(2.0 ** int(r.integers(-2, 3)))

    a_layers = _layers(2, m=512, shapes=shapes)
    a = ScheduleStep(a_layers, history_len=L)
    for t in range(cut):
        perturb(a_layers, t)
        a.run(t)
    ckpt = a.state_dict()
    saved_inputs = [[tuple(v.clone() for v in lin) for lin in layer] for layer in a_layers]
    trace_a = []
    for t in range(cut, steps):
        perturb(a_layers, t)
        a.run(t)
        trace_a.append({k: getattr(a.fwd, k).clone() for k in a.fwd.FIELDS})
    # a fresh schedule on the saved inputs, restored from the checkpoint
    b = ScheduleStep(saved_inputs, history_len=L)
    b.load_state_dict(ckpt)
    for i, t in enumerate(range(cut, steps)):
        perturb(saved_inputs, t)
        b.run(t)
        for k in b.fwd.FIELDS:
            assert torch.equal(getattr(b.fwd, k), trace_a[i][k]), (t, k)
    for k in a.bwd.FIELDS:
        assert torch.equal(getattr(a.bwd, k), getattr(b.bwd, k)), k
    with pytest.raises(ValueError):
        ScheduleStep(saved_inputs, history_len=8).load_state_dict(ckpt)
    G.check_no_device_error()
