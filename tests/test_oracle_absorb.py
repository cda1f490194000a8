"""Pins of the oracle's per-head contractions around the attention core ("vllm.models.
kimi_k3.nvidia.mla": BMM1 of the decode query with W_UK_T in _attention, the W_UV
up-projection in _v_up_proj, the sigmoid output gate of forward): against torch's batched
matmul in fp64 on the same bf16 values, per-head independence, and the gate's closed forms."""
import numpy as np
import torch

from mla_latent_cache_attention_gb300 import synth


def f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def data(seed, B, H, K, F):
    rng = np.random.default_rng(seed)
    return synth.normal_bf16_bits(rng, (B, H, K)), synth.normal_bf16_bits(rng, (H, K, F)), rng


def test_matches_torch_bmm(orc):
    x, w, _ = data(0, 5, 3, 128, 512)
    y = orc.head_bmm(x, w)
    ref = torch.bmm(f64(x).transpose(0, 1), f64(w)).transpose(0, 1).numpy()   # (H,B,K) x (H,K,F)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-12)


def test_heads_are_independent_and_strided_input(orc):
    x, w, _ = data(1, 4, 3, 64, 128)
    big = np.zeros((4, 3, 80), dtype=np.uint16)
    big[:, :, :64] = x
    y = orc.head_bmm(big[:, :, :64], w)
    w2 = w.copy()
    w2[1] = 0
    y2 = orc.head_bmm(x, w2)
    assert np.array_equal(y[:, [0, 2]], y2[:, [0, 2]]) and np.all(y2[:, 1] == 0)
    # one-hot input picks the weight row
    e = np.zeros((1, 3, 64), dtype=np.uint16)
    e[0, :, 7] = 0x3F80                                                          # bf16 1.0
    np.testing.assert_array_equal(orc.head_bmm(e, w)[0], f64(w)[:, 7, :].numpy())


def test_gate(orc):
    x, w, rng = data(2, 3, 2, 64, 128)
    y = orc.head_bmm(x, w)
    zero = np.zeros((3, 2 * 128), dtype=np.uint16)                               # sigmoid(0) = 1/2
    np.testing.assert_array_equal(orc.head_bmm(x, w, zero), 0.5 * y)
    g = synth.normal_bf16_bits(rng, (3, 256))
    sg = 1.0 / (1.0 + np.exp(-f64(g).numpy().reshape(3, 2, 128)))
    np.testing.assert_allclose(orc.head_bmm(x, w, g), y * sg, rtol=1e-14, atol=1e-14)
