"""iha_forward_noalloc: the forward pass for callers that cannot allocate device
memory (their GPU memory is already reserved by another framework's pool, or
they run where an allocation must not happen).  Its workspace is a fixed array
inside the library.

Both entry points run the same kernels on the same inputs, so the output of
iha_forward_noalloc must equal iha_forward_ex's bit for bit; a scratch-aliasing
error of any size would break that.  Two calls in a row, of different problems,
make the second run on the contents the first left behind.  The first problem is
also checked against the fp64 oracle at the bf16 tolerance of the parity tests.
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import iha_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

BF16_RMS_TOL = 2e-2


@pytest.fixture(scope="module")
def iha():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_variant_gb300 as m
    return m


def call_pair(iha, w, inp):
    """(output of iha_forward_noalloc, output of iha_forward_ex) for workload w, on the CPU."""
    d = {k: v.to("cuda:0").contiguous() for k, v in inp.items()}
    dt = iha.IHA_DTYPE_BF16 if w.dtype == "bf16" else iha.IHA_DTYPE_F32
    args = (d["X"], d["W_Q"], d["W_K"], d["W_V"], d["alpha_Q"], d["alpha_K"], d["alpha_V"], d["R"],
            w.B, w.N, w.H, w.d, w.P, w.mask_mode, w.window)
    stream = torch.cuda.current_stream()
    out_na = torch.full_like(d["X"], float("nan"))
    iha.check(iha.iha_forward_noalloc(*args, out_na, dt, stream), "iha_forward_noalloc")
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status(stream)
    assert rc == iha.IHA_OK, f"device status {rc} ({code:#x})"
    nbytes = iha.iha_workspace_bytes(w.B, w.N, w.H, w.d, w.P, dt)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:0")
    out_ex = torch.empty_like(d["X"])
    iha.check(iha.iha_forward_ex(*args, out_ex, dt, stream, ws, nbytes), "iha_forward_ex")
    torch.cuda.synchronize()
    return out_na.cpu(), out_ex.cpu()


def test_noalloc_matches_forward_ex_twice_in_a_row(iha):
    first = gi.Workload("noalloc_a", B=2, N=300, H=4, d=128, P=2, mask_mode=gi.MASK_CAUSAL, window=0,
                        dtype="bf16", seed=61)
    second = gi.Workload("noalloc_b", B=1, N=257, H=3, d=64, P=3, mask_mode=gi.MASK_WINDOW, window=20,
                         dtype="bf16", seed=62)
    for k, w in enumerate((first, second)):
        inp = gi.make_inputs(w)
        got, ref = call_pair(iha, w, inp)
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref), f"{w.name}: iha_forward_noalloc differs from iha_forward_ex"
        if k == 0:
            f = gi.as_f64(inp)
            o = oracle.forward(f["X"], f["W_Q"], f["W_K"], f["W_V"], f["alpha_Q"], f["alpha_K"], f["alpha_V"],
                               f["R"], H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window)
            g = got.double().numpy().reshape(o.shape)
            e = float(np.sqrt(np.mean((g - o) ** 2)) / np.sqrt(np.mean(o ** 2)))
            assert e <= BF16_RMS_TOL, f"{w.name}: RMS(err)/RMS(O) = {e:.3e} against the oracle"


def test_noalloc_refuses_problems_larger_than_its_array(iha):
    w = gi.WORKLOADS["bf16_window1024_n4096"]
    assert iha.iha_workspace_bytes(w.B, w.N, w.H, w.d, w.P, iha.IHA_DTYPE_BF16) > iha.IHA_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20   # never dereferenced: the size check comes first
    rc = iha.iha_forward_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, w.B, w.N, w.H, w.d, w.P,
                                 w.mask_mode, w.window, fake, iha.IHA_DTYPE_BF16, None)
    assert rc == iha.IHA_ERR_WORKSPACE
