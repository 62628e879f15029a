"""Host <-> device conversions shared by the GPU tests (no routing arithmetic)."""
import numpy as np
import torch


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_host(t: torch.Tensor) -> np.ndarray:
    """CUDA tensor -> numpy; bf16 comes back as uint16 bit patterns."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def misaligned_like(a: torch.Tensor, offset_elems: int = 1) -> torch.Tensor:
    """A contiguous copy of ``a`` whose data pointer is offset by a few elements."""
    buf = torch.empty(a.numel() + offset_elems, dtype=a.dtype, device=a.device)
    view = buf[offset_elems:].view(a.shape)
    view.copy_(a)
    return view


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        g, w = got.view(np.uint32), want.view(np.uint32)
    else:
        g, w = got, want
    bad = np.flatnonzero(g.reshape(-1) != w.reshape(-1))
    assert bad.size == 0, "%s: %d of %d elements differ, first at %d: got %r want %r" % (
        what, bad.size, g.size, bad[0], got.reshape(-1)[bad[0]], want.reshape(-1)[bad[0]])


def f32(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a


def assert_close_fp32(got: np.ndarray, want: np.ndarray, what: str, rtol: float = 1e-5):
    """max abs error <= rtol * (1 + |ref|), element by element."""
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    lim = rtol * (1.0 + np.abs(want.astype(np.float64)))
    bad = np.flatnonzero(~(err <= lim))
    assert bad.size == 0, "%s: %d elements outside tolerance, worst err %g at %d (ref %g)" % (
        what, bad.size, err.reshape(-1)[bad].max(), bad[0], want.reshape(-1)[bad[0]])


def assert_close_bf16(got: np.ndarray, want: np.ndarray, what: str, rel: float = 2e-2):
    """bf16 outputs: |got - ref| <= rel * max(|ref|, tiny)."""
    g, w = f32(got).astype(np.float64), f32(want).astype(np.float64)
    err = np.abs(g - w)
    bad = np.flatnonzero(~(err <= rel * np.maximum(np.abs(w), 1e-30)) & ~(err == 0))
    assert bad.size == 0, "%s: %d bf16 elements outside %g relative" % (what, bad.size, rel)
