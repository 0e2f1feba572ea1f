"""The seeded input recipe: deterministic, slice-regenerable, with the stated distributions."""
import math

import numpy as np

import workloads as W


def test_slices_are_deterministic_and_independent():
    w = W.WORKLOADS["decode_b64_l36_t1"]
    a = W.sequence_slice(w, 3, 7)
    b = W.sequence_slice(w, 3, 7)
    c = W.sequence_slice(w, 7, 3)
    for k in a:
        assert np.array_equal(a[k], b[k])
        assert not np.array_equal(a[k], c[k])
    assert np.array_equal(W.layer_weights(w, 5)["conv_w"], W.layer_weights(w, 5)["conv_w"])


def test_host_inputs_equal_slices():
    w = W.WORKLOADS["verify_b16_l36_t8_ragged"].scaled(B=3, L=2)
    h = W.host_inputs(w, threads=4)
    for b in range(3):
        for l in range(2):
            sl = W.sequence_slice(w, b, l)
            for k, v in sl.items():
                assert np.array_equal(h[k][b, l], v)
    for l in range(2):
        for k, v in W.layer_weights(w, l).items():
            assert np.array_equal(h[k][l], v)
    assert h["seq_len"].dtype == np.int32 and h["seq_len"].shape == (3,)


def test_distributions():
    w = W.WORKLOADS["decode_b64_l36_t1"]
    sl = W.sequence_slice(w, 0, 0)
    wt = W.layer_weights(w, 0)
    assert abs(sl["state"].std() - 0.05) < 0.001 and abs(sl["state"].mean()) < 0.001
    assert abs(sl["conv_state"].std() - 1.0) < 0.02
    assert abs(wt["conv_w"].std() - 0.25) < 0.005
    assert abs(wt["ssm_norm"].mean() - 1.0) < 0.03
    assert np.all(wt["ssm_a"] <= -1.0) and np.all(wt["ssm_a"] >= -16.0)
    lg = np.log(-W.layer_weights(w, 1)["ssm_a"].astype(np.float64))
    assert 0.0 <= lg.min() and lg.max() <= math.log(16.0)
    hi = W.WORKLOADS["decode_b128_l36_t1_beta_hi_decay_hi"]
    s3 = W.sequence_slice(hi, 1, 1)
    assert abs(s3["beta"].mean() - 2.0) < 0.4 and abs(s3["alpha"].mean() + 2.0) < 0.4
    z = W.sequence_slice(W.WORKLOADS["decode_b1_l36_t64_zero_state"], 0, 4)
    assert np.all(z["state"] == 0.0) and z["qkv"].shape == (64, 10240)
    lens = W.seq_lens(W.WORKLOADS["verify_b16_l36_t8_ragged"])
    assert lens.min() >= 1 and lens.max() <= 8 and len(set(lens.tolist())) > 2
    assert W.seq_lens(w) is None


def test_bf16_rounding_is_nearest_even_and_decodes_exactly():
    vals = np.array([1.0, -2.0, 1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20, 3.140625, 0.0, -0.0], np.float32)
    bits = W.to_bf16_bits(vals)
    assert bits.tolist() == [0x3F80, 0xC000, 0x3F80, 0x3F82, 0x3F81, 0x4049, 0x0000, 0x8000]
    back = W.bf16_bits_to_float(bits)
    assert back.tolist() == [1.0, -2.0, 1.0, 1 + 2**-6, 1 + 2**-7, 3.140625, 0.0, -0.0]


def test_projection_head_streams_are_independent_and_scaled():
    w = W.WORKLOADS["decode_b1_l1_t1"]
    a = W.proj_head_weights(w, "w_qkv", 0, 5, n_embd=256)
    b = W.proj_head_weights(w, "w_qkv", 0, 6, n_embd=256)
    g = W.proj_head_weights(w, "w_gate", 0, 5, n_embd=256)
    assert a.shape == (128, 256) and a.dtype == np.uint16
    assert not np.array_equal(a, b) and not np.array_equal(a, g)
    full = W.proj_weights(w, 0, n_embd=256)
    assert full["w_qkv"].shape == (10240, 256) and full["w_gate"].shape == (6144, 256)
    assert np.array_equal(full["w_qkv"][640:768], a) and np.array_equal(full["w_gate"][640:768], g)
    std = W.bf16_bits_to_float(full["w_qkv"]).std()
    assert abs(std * 16.0 - 1.0) < 0.01
