"""Helpers shared by the GPU parity tests: host <-> device marshalling and the tolerance
checks (attention: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| elementwise, lse within 1e-3
absolute; inserts, concat and gathers: bit-exact)."""
import numpy as np
import torch

ATOL, RTOL, LSE_TOL = 1e-2, 1e-2, 1e-3


def dev():
    return torch.device("cuda", 0)


def t_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def t_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def t_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def t_i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev())


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_attn_close(out_gpu: torch.Tensor, ref: np.ndarray, what=""):
    o = out_gpu.float().cpu().numpy()
    assert o.shape == ref.shape, (o.shape, ref.shape)
    err = np.abs(o - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {i.tolist()}: "
                             f"gpu {o[tuple(i[0])]} oracle {ref[tuple(i[0])]}; max err {err.max()}")


def assert_lse_close(lse_gpu: torch.Tensor, ref: np.ndarray, what="", rel=0.0):
    """|lse_gpu - lse_oracle| <= LSE_TOL (+ rel * |lse_oracle| where a test's logits are so
    large that fp32 itself cannot resolve 1e-3: one fp32 ulp at 3e4 is 2e-3)."""
    l = lse_gpu.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: -inf pattern differs"
    assert np.all(l[~fin] == -np.inf), f"{what}: empty rows must give -inf"
    if fin.any():
        err = np.abs(l[fin] - ref[fin])
        assert np.all(err <= LSE_TOL + rel * np.abs(ref[fin])), f"{what}: lse max err {err.max()}"
