"""The seeded generator: deterministic, order-independent, and drawing the stated distributions."""
import numpy as np

import oracle
import synth


def test_deterministic_and_sliceable():
    a = synth.gen_x(0, 64, 256, threads=1)
    b = synth.gen_x(0, 64, 256, threads=8)
    assert np.array_equal(a, b)
    att = np.zeros(64, np.int32)
    att[5] = 3
    c = synth.gen_x(0, 64, 256, att)
    assert np.array_equal(np.delete(c, 5, 0), np.delete(a, 5, 0)) and not np.array_equal(c[5], a[5])
    w1, s1 = synth.gen_mxfp4(0, 4, 9, 64, 256, 256)
    w2, s2 = synth.gen_mxfp4(0, 4, 9, 32, 256, 256, row0=32)
    assert np.array_equal(w1[32:], w2) and np.array_equal(s1[32:], s2)


def test_x_is_standard_normal_bf16():
    x = synth.gen_x(1, 256, 1024)
    v = np.array([oracle.bf16_value(int(h)) for h in x.reshape(-1)[:20000]])
    assert abs(v.mean()) < 0.03 and abs(v.std() - 1) < 0.03


def test_expert_weights_look_like_n01_over_d():
    d = 4096
    ex = synth.gen_experts(0, 2, d, 2048)
    v = oracle.mxfp4_dequantize(ex.w13[0, :64], ex.s13[0, :64])
    assert abs(v.std() * np.sqrt(d) - 1.0) < 0.15
    assert set(np.unique(ex.s13)) <= {127 + synth._lib().synth_weight_e0(d), 126 + synth._lib().synth_weight_e0(d)}


def test_router_and_hot_bias():
    w, b, hot = synth.gen_router(0, 256, 4096, n_hot=26)
    assert w.dtype == np.float32 and abs(w.std() * 64 - 1) < 0.01
    assert len(set(hot.tolist())) == 26
    assert np.all(b[hot] > 0.89) and np.all(np.abs(np.delete(b, hot)) <= 0.1)
