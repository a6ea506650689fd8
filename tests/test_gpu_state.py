"""GPU parity of delayed scaling (amax history 16 over 32 steps: casts with the
previous scale, records the amax, updates the history) and the failure paths
(a bounded wait that runs out, a state argument out of range) -- none of which
faults or hangs the GPU."""
import numpy as np
import pytest
import torch

import oracle
import scaled_quantize_gemm_amax_gb300 as fq
from scaled_quantize_gemm_amax_gb300 import workloads as wl
from gpu_util import R, F, assert_bytes_equal, assert_status_ok, bits16, f32bits, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _step_inputs(step, fin=1024, tokens=256):
    x = wl.normal_bf16((tokens, fin), wl.seed_of(4, wl.ROLE_X, step), 1.0)
    if step == wl.CFG4_SPIKE_STEP:
        x = (x.float() * wl.CFG4_SPIKE).to(torch.bfloat16)
    dy = wl.normal_bf16((tokens, fin), wl.seed_of(4, wl.ROLE_DY, step), 1e-3)
    return x, dy


def _run_delayed(steps, st_x, st_dy, ref_x, ref_dy, start=0):
    for t in range(start, start + steps):
        x, dy = _step_inputs(t)
        for x_t, st, ref, fmt in ((x, st_x, ref_x, F.E4M3), (dy, st_dy, ref_dy, F.E5M2)):
            xh = bits16(x_t)
            # cast with the current (previous-step) scale, recording this step's amax
            qr, _, qc, _ = fq.cast_transpose(x_t, R.TENSOR, fmt, st.scale, st.amax)
            st.update()
            torch.cuda.synchronize()
            assert_status_ok()
            q_ref, _ = oracle.quantize_rowwise(xh, oracle.KIND_TENSOR, int(fmt), ref.scale[0])
            assert_bytes_equal(host(qr), q_ref, f"step {t} q_row")
            assert_bytes_equal(host(qc), np.ascontiguousarray(q_ref.T), f"step {t} q_col")
            ref.step(oracle.amax(xh))
            assert_bytes_equal(f32bits(host(st.hist)), f32bits(ref.hist), f"step {t} hist")
            assert host(st.pos)[0] == ref.pos[0]
            assert f32bits(host(st.scale))[0] == f32bits(ref.scale[0]), f"step {t} scale"
            assert f32bits(host(st.scale_inv))[0] == f32bits(ref.scale_inv[0]), f"step {t} scale_inv"


def test_delayed_scaling_32_steps_bit_exact():
    st_x, st_dy = fq.DelayedScaling(16, F.E4M3), fq.DelayedScaling(16, F.E5M2)
    ref_x, ref_dy = oracle.DelayedState(16, oracle.E4M3), oracle.DelayedState(16, oracle.E5M2)
    _run_delayed(32, st_x, st_dy, ref_x, ref_dy)


def test_delayed_scaling_checkpoint_resume():
    st_x, st_dy = fq.DelayedScaling(16, F.E4M3), fq.DelayedScaling(16, F.E5M2)
    ref_x, ref_dy = oracle.DelayedState(16, oracle.E4M3), oracle.DelayedState(16, oracle.E5M2)
    _run_delayed(16, st_x, st_dy, ref_x, ref_dy)
    saved = (st_x.state_dict(), st_dy.state_dict())
    # fresh buffers, restored state, then the remaining 16 steps must match the oracle
    new_x, new_dy = fq.DelayedScaling(16, F.E4M3), fq.DelayedScaling(16, F.E5M2)
    new_x.load_state_dict(saved[0])
    new_dy.load_state_dict(saved[1])
    _run_delayed(16, new_x, new_dy, ref_x, ref_dy, start=16)


def test_history_position_out_of_range_is_reported():
    st = fq.DelayedScaling(16, F.E4M3)
    st.pos.fill_(99)
    st.amax.fill_(2.0)
    before = host(st.hist).copy()
    st.update()
    assert fq.fp8_get_device_status() == fq.Status.ERR_DEVICE_STATE
    assert np.array_equal(host(st.hist), before) and host(st.pos)[0] == 99
    assert fq.fp8_get_device_status() == fq.Status.OK     # the word was cleared


def test_bounded_wait_times_out_and_context_survives():
    fq.fp8_debug_wait_timeout()
    assert fq.fp8_get_device_status() == fq.Status.ERR_TIMEOUT
    # the context is still usable
    x = wl.normal_bf16((128, 128), 7)
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    fq.fp8_amax(x, amax)
    torch.cuda.synchronize()
    assert f32bits(host(amax))[0] == f32bits(oracle.amax(bits16(x)))
    assert_status_ok()


def test_delayed_scaling_gpt175b_qkv_full_size():
    # The GPT-175B QKV linear's X [2048, 12288] (E4M3) and dY [2048, 36864] (E5M2) over 32
    # steps with the x10 spike at step 8, at full size: amax, history, position, scale and
    # scale_inv bit for bit every step; the FP8 bytes on seeded rows of both copies.
    st = {"x": fq.DelayedScaling(16, F.E4M3), "dy": fq.DelayedScaling(16, F.E5M2)}
    ref = {"x": oracle.DelayedState(16, oracle.E4M3), "dy": oracle.DelayedState(16, oracle.E5M2)}
    rng = np.random.default_rng(4100)
    for t in range(32):
        x, _, dy = wl.cfg4_step("qkv", t)
        for key, x_t, fmt in (("x", x, F.E4M3), ("dy", dy, F.E5M2)):
            rows, cols = x_t.shape
            qr, _, qc, _ = fq.cast_transpose(x_t, R.TENSOR, fmt, st[key].scale, st[key].amax)
            st[key].update()
            torch.cuda.synchronize()
            assert_status_ok()
            xh = bits16(x_t)
            r = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 30, replace=False)]))
            c = np.unique(np.concatenate([[0, cols - 1], rng.choice(cols, 30, replace=False)]))
            q_r, _ = oracle.quantize_rowwise(xh[r], oracle.KIND_TENSOR, int(fmt), ref[key].scale[0])
            q_c, _ = oracle.quantize_rowwise(np.ascontiguousarray(xh[:, c].T), oracle.KIND_TENSOR, int(fmt),
                                             ref[key].scale[0])
            assert_bytes_equal(host(qr[torch.as_tensor(r, device=qr.device)]), q_r, f"step {t} {key} q_row")
            assert_bytes_equal(host(qc[torch.as_tensor(c, device=qc.device)]), q_c, f"step {t} {key} q_col")
            ref[key].step(oracle.amax(xh))
            assert_bytes_equal(f32bits(host(st[key].hist)), f32bits(ref[key].hist), f"step {t} {key} hist")
            assert host(st[key].pos)[0] == ref[key].pos[0]
            assert f32bits(host(st[key].scale))[0] == f32bits(ref[key].scale[0]), f"step {t} {key} scale"
            assert f32bits(host(st[key].scale_inv))[0] == f32bits(ref[key].scale_inv[0]), f"step {t} {key} scale_inv"
