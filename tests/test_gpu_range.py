"""FP16 operand range guard (include/kvq.h, conventions): an attention call
whose rotated query, rotated current values, cached key step sizes or cached
values leave the range of the FP16 tensor-core operands still completes, but
records KVQ_ERR_RANGE in the device status word instead of returning inf/NaN
silently; the next in-range call reads KVQ_OK again.  Ordinary inputs and a
status read: nothing here faults."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_quantize_gb300 import kvq, synth
from tests.gpu_common import assert_close, build_cache, oracle_head

pytestmark = pytest.mark.gpu


def _setup(bits=2, group=32, seed=7):
    w = synth.Workload("range", heads=2, head_dim=128, chunk_tokens=128, n_chunks=2, bits=bits,
                       group=group, n_outliers_fixed=2, outlier_scale=6.0)
    x = synth.inputs(w, seed=seed, n_q=130, n_s=256, n_r=100)
    s = synth.hadamard_signs(128, seed=seed)
    return w, x, s


def _status_after(cache, x, corr=kvq.CORR_TAYLOR):
    kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(), x["v_cur"].cuda(), corr=corr,
                            with_mass=True)
    torch.cuda.synchronize()
    return kvq.last_device_status()


def _in_range_call_is_ok_again(w, x, s):
    cache = build_cache(w, x, s)
    out, ps, pr = kvq.attention_corrected(cache, x["q"].cuda(), x["k_cur"].cuda(),
                                          x["v_cur"].cuda(), with_mass=True)
    torch.cuda.synchronize()
    assert kvq.last_device_status() == kvq.KVQ_OK
    o_ref, ps_ref, pr_ref = oracle_head(w, x, s, 0, 1, np.arange(x["q"].shape[2]), 1)
    assert_close(out[0, 1].float().cpu().numpy(), o_ref, ps[0, 1].cpu().numpy(), ps_ref,
                 pr[0, 1].cpu().numpy(), pr_ref, what="after a range error")


def test_query_beyond_fp16_after_rotation():
    w, x, s = _setup()
    cache = build_cache(w, x, s)
    bad = dict(x)
    q = x["q"].clone()
    q[0, 1, 17, 5] = 1.0e6        # rotated: 1e6 / sqrt(128) ~ 8.8e4 > 65504 in every channel
    bad["q"] = q
    assert _status_after(cache, bad) == kvq.KVQ_ERR_RANGE
    _in_range_call_is_ok_again(w, x, s)


def test_current_values_beyond_fp16_after_rotation():
    w, x, s = _setup()
    cache = build_cache(w, x, s)
    bad = dict(x)
    v = x["v_cur"].clone()
    v[0, 0, 3, 64] = -2.0e6
    bad["v_cur"] = v
    assert _status_after(cache, bad) == kvq.KVQ_ERR_RANGE
    _in_range_call_is_ok_again(w, x, s)


@pytest.mark.parametrize("bits,group", [(2, 32), (4, 64)])
def test_key_step_beyond_the_fp16_key_constant(bits, group):
    """One cached key row spans ~5.3e4 after rotation: its step size exceeds
    65504 / 16 (INT2, g32: ~1.8e4) and 65504 / 24 (INT4, g64: ~3.5e3)."""
    w, x, s = _setup(bits, group)
    bad = dict(x)
    k = x["k_win"].clone()
    k[0, 0, 40, 9] = 3.0e5
    bad["k_win"] = k
    cache = build_cache(w, bad, s)
    assert _status_after(cache, bad) == kvq.KVQ_ERR_RANGE
    _in_range_call_is_ok_again(w, x, s)


def test_cached_value_beyond_fp16():
    w, x, s = _setup()
    bad = dict(x)
    v = x["v_win"].clone()
    v[0, 1, 200, 0] = 3.0e6       # rotated ~2.6e5 per channel: (|z| + 3) D > 65504
    bad["v_win"] = v
    cache = build_cache(w, bad, s)
    assert _status_after(cache, bad) == kvq.KVQ_ERR_RANGE
    _in_range_call_is_ok_again(w, x, s)


def test_per_channel_taylor_query_limit():
    """Per-channel keys with the Taylor term square the rotated query in
    FP16 (q'^2 / 64): |q'| >= 2047 is out of range there, fine otherwise."""
    w, x, s = _setup()
    cache = kvq.KVCache(1, 2, 128, 2, 32, 128, 2, s, key_mode=kvq.KEYS_PER_CHANNEL)
    kvq.quantize_append(cache, x["k_win"][:, :, :128].cuda().contiguous(),
                        x["v_win"][:, :, :128].cuda().contiguous())
    bad = dict(x)
    q = x["q"].clone()
    q[0, 0, 2, 100] = 4.0e4       # rotated ~3.5e3 per channel: > 2047, < 65504
    bad["q"] = q
    assert _status_after(cache, bad, corr=kvq.CORR_TAYLOR) == kvq.KVQ_ERR_RANGE
    assert _status_after(cache, bad, corr=kvq.CORR_NONE) == kvq.KVQ_OK
