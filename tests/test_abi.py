"""The C-ABI library loads, exports every symbol include/iha.h declares, and its
host-side logic (validation, sizes, error strings) behaves as documented.
No call here reaches the GPU: every compute call below is rejected during
argument validation, before anything is launched."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def iha():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import transformer_attention_variant_gb300 as m
    return m


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "iha.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(iha_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(iha):
    syms = declared_symbols()
    assert len(syms) >= 12
    lib = ctypes.CDLL(iha.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), f"libiha.so does not export {s}"
    assert sorted(iha.EXPORTED) == syms


def test_binding_has_the_abi_names(iha):
    for s in declared_symbols():
        assert callable(getattr(iha, s)), s


def test_error_strings(iha):
    assert iha.iha_error_string(iha.IHA_OK) == "ok"
    assert "invalid" in iha.iha_error_string(iha.IHA_ERR_INVALID_ARG)
    assert "timed out" in iha.iha_error_string(iha.IHA_ERR_TIMEOUT)
    assert "rebuild" in iha.iha_error_string(iha.IHA_ERR_BUILD)
    assert iha.iha_error_string(12345) == "unknown status"


def test_workspace_bytes(iha):
    B, N, H, d, P = 2, 1024, 16, 64, 2
    D = H * d
    al = lambda x: (x + 255) // 256 * 256
    for dtype, es in ((iha.IHA_DTYPE_BF16, 2), (iha.IHA_DTYPE_F32, 4)):
        # first region: folded weights, or the slice-major weights on the unfolded route
        # (W_Q, W_K, W_V reordered: 3 D x D, no padding at 16 heads)
        first = 3 * D * D * es if iha.iha_projection_route(H, d, P, dtype) == 1 else 3 * H * P * d * D * es
        # + the 256-byte control slot (the call's attention work counter)
        expect = al(first) + al(3 * B * H * N * P * d * es) + al(B * N * H * P * d * es) + 256
        assert iha.iha_workspace_bytes(B, N, H, d, P, dtype) == expect
    assert iha.iha_workspace_bytes(0, N, H, d, P, 1) == 0
    assert iha.iha_workspace_bytes(B, N, H, 96, P, 1) == 0       # bf16 needs d in {64, 128}
    assert iha.iha_workspace_bytes(B, N, H, 96, P, 0) > 0        # fp32 takes any d <= 256
    assert iha.iha_workspace_bytes(B, N, H, d, P, 7) == 0
    assert iha.iha_host_buffer_bytes(B, N, H, d, P, 1) > iha.iha_workspace_bytes(B, N, H, d, P, 1)


FAKE = 1 << 20   # a non-null address that is never dereferenced (validation fails first)


def fwd(iha, **kw):
    a = dict(X=FAKE, W_Q=FAKE, W_K=FAKE, W_V=FAKE, alpha_Q=FAKE, alpha_K=FAKE, alpha_V=FAKE, R=FAKE,
             B=1, N=8, H=2, d=64, P=2, mask_mode=1, window=0, out=FAKE, dtype=1, stream=None,
             workspace=None, workspace_bytes=0)
    a.update(kw)
    return iha.iha_forward_ex(**a)


@pytest.mark.parametrize("kw,status", [
    (dict(X=None), 1), (dict(out=None), 1), (dict(R=None), 1), (dict(alpha_V=None), 1),
    (dict(B=0), 1), (dict(N=-1), 1), (dict(H=0), 1), (dict(P=0), 1), (dict(d=0), 1),
    (dict(mask_mode=3), 1), (dict(mask_mode=-1), 1), (dict(mask_mode=2, window=0), 1),
    (dict(dtype=2), 1), (dict(d=96), 2), (dict(d=32), 2), (dict(dtype=0, d=300), 2),
    (dict(N=1 << 24, P=2), 2),
    (dict(workspace=FAKE, workspace_bytes=16), 3),
    (dict(workspace=FAKE + 8, workspace_bytes=1 << 40), 3),
])
def test_forward_rejects_bad_arguments(iha, kw, status):
    assert fwd(iha, **kw) == status


def test_projection_route(iha):
    assert iha.iha_projection_route(16, 128, 4, iha.IHA_DTYPE_BF16) == 1
    assert iha.iha_projection_route(16, 64, 2, iha.IHA_DTYPE_BF16) == 1
    assert iha.iha_projection_route(16, 128, 1, iha.IHA_DTYPE_BF16) == 1
    assert iha.iha_projection_route(32, 64, 2, iha.IHA_DTYPE_BF16) == 0
    assert iha.iha_projection_route(4, 32, 2, iha.IHA_DTYPE_F32) == 0
    assert iha.iha_projection_route(4, 96, 2, iha.IHA_DTYPE_BF16) == -1


def test_step_entry_points_reject_bad_arguments(iha):
    assert iha.iha_project_heads(FAKE, None, FAKE, FAKE, 1, 8, 2, 64, 1, FAKE) == 1
    assert iha.iha_project_heads(FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 0, FAKE) == 2
    assert iha.iha_mix_heads(FAKE, FAKE, FAKE, FAKE, 1, 8, 32, 64, 2, 1, FAKE) == 2
    assert iha.iha_mix_heads(FAKE, FAKE, FAKE, None, 1, 8, 2, 64, 2, 1, FAKE) == 1
    assert iha.iha_project_mix(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 64, 2, 1, FAKE) == 1
    assert iha.iha_project_mix(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 32, 64, 2, 1, FAKE) == 2   # H > 16
    assert iha.iha_project_mix(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 2, 0, FAKE) == 2    # fp32
    assert iha.iha_project_mix(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 2, 1, FAKE + 16) == 1   # QKV not 32-aligned
    assert iha.iha_slice_weights(FAKE, None, FAKE, 2, 64, 1, FAKE) == 1
    assert iha.iha_slice_weights(FAKE, FAKE, FAKE, 32, 64, 1, FAKE) == 2
    assert iha.iha_sliced_weights_bytes(16, 128, 1) == 3 * 2048 * 2048 * 2   # 16 heads: no padding
    assert iha.iha_sliced_weights_bytes(5, 64, 1) == 3 * 320 * 2 * 192 * 2   # 5 x 32 columns padded to 192
    assert iha.iha_sliced_weights_bytes(16, 128, 0) == 0
    assert iha.iha_fold_weights(None, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 64, 2, 1, FAKE) == 1
    assert iha.iha_project(FAKE, FAKE, 1, 8, 2, 64, 0, 1, FAKE) == 1
    assert iha.iha_attention(FAKE, 1, 8, 2, 64, 2, 2, 0, 1, FAKE) == 1
    assert iha.iha_attention(FAKE, 1, 8, 2, 48, 2, 1, 0, 1, FAKE) == 2
    assert iha.iha_attention(FAKE, 1, 8, 2, 64, 2, 1, 0, 1, FAKE + 2) == 1    # Pbar not 16-aligned
    assert iha.iha_attention(FAKE + 8, 1, 8, 2, 64, 2, 1, 0, 1, FAKE) == 1    # QKV not 16-aligned
    assert iha.iha_contract(FAKE, None, 1, 8, 2, 64, 2, 1, FAKE) == 1
    assert iha.iha_forward(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 2, 1, 0, FAKE) == 1
    assert iha.iha_forward_host(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 2, 5, 0, FAKE, 1) == 1
    assert iha.iha_selftest_wait_timeout(None, 0) == 1
    assert iha.iha_selftest_wait_timeout(None, 20000) == 1


def test_host_buffer_layout_and_checks(iha):
    """iha_host_buffer_bytes is X, W_Q, W_K, W_V, alpha_Q/K/V, R and out (each from a
    256-byte boundary) followed by iha_forward_ex's workspace; iha_forward_host refuses a
    caller-given device buffer that is smaller or not 256-byte aligned before any copy."""
    al = lambda x: (x + 255) // 256 * 256
    bf16 = iha.IHA_DTYPE_BF16
    for B, N, H, d, P in ((1, 64, 2, 64, 2), (2, 100, 16, 128, 4), (1, 33, 5, 64, 3), (3, 7, 16, 128, 1)):
        D = H * d
        x, w, a = B * N * D * 2, D * D * 2, H * H * P * 4
        expect = al(x) + 3 * al(w) + 4 * al(a) + al(x) + iha.iha_workspace_bytes(B, N, H, d, P, bf16)
        need = iha.iha_host_buffer_bytes(B, N, H, d, P, bf16)
        assert need == expect, (B, N, H, d, P)
        args = [FAKE] * 8 + [B, N, H, d, P, 1, 0, FAKE, bf16, None]
        assert iha.iha_forward_host(*args, FAKE * 2, need - 1) == iha.IHA_ERR_WORKSPACE
        assert iha.iha_forward_host(*args, FAKE * 2 + 128, need) == iha.IHA_ERR_WORKSPACE
    assert iha.iha_host_buffer_bytes(1, 64, 2, 96, 2, bf16) == 0     # bf16 needs d in {64, 128}
    assert iha.iha_host_buffer_bytes(0, 64, 2, 64, 2, bf16) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    """Importing the binding when libiha.so is absent raises, naming the fix;
    there is no fallback path."""
    import subprocess
    import sys
    import shutil
    pkg = tmp_path / "transformer_attention_variant_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "transformer_attention_variant_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import transformer_attention_variant_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libiha.so is missing" in r.stderr


def test_stack_workspace_and_validation(iha):
    B, N, H, d = 1, 512, 4, 64
    P = [2, 2, 2, 2, 1]
    act = (B * N * H * d * 2 + 255) // 256 * 256
    expect = 2 * act + max(iha.iha_workspace_bytes(B, N, H, d, p, 1) for p in P)
    assert iha.iha_stack_workspace_bytes(P, B, N, H, d, 1) == expect
    assert iha.iha_stack_workspace_bytes([], B, N, H, d, 1) == 0
    assert iha.iha_stack_workspace_bytes([2, 0], B, N, H, d, 1) == 0          # a layer with P = 0
    fake = 1 << 40                                                           # never dereferenced
    layer = dict(W_Q=fake, W_K=fake, W_V=fake, alpha_Q=fake, alpha_K=fake, alpha_V=fake, R=fake,
                 P=2, mask_mode=2, window=32)
    ok = [dict(layer) for _ in range(5)]
    bad_p = [dict(layer), dict(layer, P=0)]
    bad_window = [dict(layer), dict(layer, window=0)]
    null_w = [dict(layer), dict(layer, W_K=None)]
    for layers, status in ((bad_p, iha.IHA_ERR_INVALID_ARG), (bad_window, iha.IHA_ERR_INVALID_ARG),
                           (null_w, iha.IHA_ERR_INVALID_ARG)):
        assert iha.iha_forward_stack(fake, layers, B, N, H, d, 1, fake) == status
    assert iha.iha_forward_stack(fake, [], B, N, H, d, 1, fake) == iha.IHA_ERR_INVALID_ARG
    assert iha.iha_forward_stack(None, ok, B, N, H, d, 1, fake) == iha.IHA_ERR_INVALID_ARG
    assert iha.iha_forward_stack(fake, ok, B, N, H, 96, 1, fake) == iha.IHA_ERR_UNSUPPORTED
    # a workspace that is too small is refused before anything runs
    assert iha.iha_forward_stack(fake, ok, B, N, H, d, 1, fake, workspace=fake, workspace_bytes=256) == \
        iha.IHA_ERR_WORKSPACE


def test_decode_validation(iha):
    fake = 1 << 40                                           # never dereferenced
    B, H, d, P = 2, 4, 64, 2
    assert iha.iha_decode_workspace_bytes(B, H, d, P) > 0
    assert iha.iha_decode_workspace_bytes(B, H, 128, 8) == 0     # d = 128 takes P <= 4
    assert iha.iha_decode_workspace_bytes(B, H, 96, 2) == 0
    args = [fake] * 8
    ok = dict(B=B, H=H, d=d, P=P, mask_mode=1, window=0, K_cache=fake, V_cache=fake, cache_tokens=100, t=5,
              out=fake, dtype=1)

    def step(**kw):
        a = dict(ok, **kw)
        return iha.iha_decode_step(*args, a["B"], a["H"], a["d"], a["P"], a["mask_mode"], a["window"],
                                   a["K_cache"], a["V_cache"], a["cache_tokens"], a["t"], a["out"], a["dtype"])
    assert step(t=100) == iha.IHA_ERR_INVALID_ARG            # no room in the cache
    assert step(t=-1) == iha.IHA_ERR_INVALID_ARG
    assert step(mask_mode=0) == iha.IHA_ERR_INVALID_ARG      # would read future tokens
    assert step(K_cache=None) == iha.IHA_ERR_INVALID_ARG
    assert step(dtype=0) == iha.IHA_ERR_UNSUPPORTED
    assert step(d=128, P=8) == iha.IHA_ERR_UNSUPPORTED
    assert step(H=64, d=64) == iha.IHA_ERR_UNSUPPORTED       # H*d > 2048
    assert step(K_cache=fake + 8) == iha.IHA_ERR_INVALID_ARG  # caches and W are read 16 bytes at a time
    assert step(V_cache=fake + 2) == iha.IHA_ERR_INVALID_ARG
    assert iha.iha_decode_step(fake, fake + 4, *args[2:], B, H, d, P, 1, 0, fake, fake, 100, 5, fake, 1) == \
        iha.IHA_ERR_INVALID_ARG
    assert iha.iha_decode_step(*args, B, H, d, P, 1, 0, fake, fake, 100, 5, fake, 1, None, fake, 16) == \
        iha.IHA_ERR_WORKSPACE
    # prefill: the cache must hold the prompt
    assert iha.iha_prefill(*args, B, 50, H, d, P, 1, 0, fake, fake, fake, 49, 1) == iha.IHA_ERR_INVALID_ARG
    assert iha.iha_prefill(*args, B, 50, H, d, P, 0, 0, fake, fake, fake, 60, 1) == iha.IHA_ERR_INVALID_ARG


def test_training_pair_validation(iha):
    fake = 1 << 40                                           # never dereferenced
    B, N, H, d, P = 2, 64, 4, 64, 2
    args = [fake] * 8
    nb = iha.iha_backward_workspace_bytes(B, N, H, d, P, 1)
    # the workspace carries the forward pieces from one call to the other: it is required
    assert iha.iha_forward_train(*args, B, N, H, d, P, 1, 0, fake, 1, None, None, 0) == iha.IHA_ERR_WORKSPACE
    assert iha.iha_backward_saved(*args, B, N, H, d, P, 1, 0, fake, *([fake] * 8), 1, None, None, 0) == \
        iha.IHA_ERR_WORKSPACE
    assert iha.iha_forward_train(*args, B, N, H, d, P, 1, 0, fake, 1, None, fake, nb - 256) == iha.IHA_ERR_WORKSPACE
    assert iha.iha_forward_train(*args, B, N, 20, d, P, 1, 0, fake, 1, None, fake, nb) == iha.IHA_ERR_UNSUPPORTED
    assert iha.iha_forward_train(*args, B, N, H, d, P, 1, 0, fake, 0, None, fake, nb) == iha.IHA_ERR_UNSUPPORTED
    assert iha.iha_forward_train(*args, B, N, H, d, P, 1, 0, None, 1, None, fake, nb) == iha.IHA_ERR_INVALID_ARG
    assert iha.iha_backward_saved(*args, B, N, H, d, P, 1, 0, fake, None, *([fake] * 7), 1, None, fake, nb) == \
        iha.IHA_ERR_INVALID_ARG


def test_backward_gradient_alignment(iha):
    fake = 1 << 40                                           # never dereferenced
    B, N, H, d, P = 2, 64, 4, 64, 2
    args = [fake] * 8
    for i in range(4):   # dX, dW_Q, dW_K, dW_V are written by TMA stores
        g = [fake] * 8
        g[i] = fake + 8
        assert iha.iha_backward(*args, B, N, H, d, P, 1, 0, fake, *g, 1) == iha.IHA_ERR_INVALID_ARG


def test_backward_validation(iha):
    fake = 1 << 40                                           # never dereferenced
    B, N, H, d, P = 2, 64, 4, 64, 2
    assert iha.iha_backward_workspace_bytes(B, N, H, d, P, 1) > 0
    assert iha.iha_backward_workspace_bytes(B, N, 20, d, P, 1) == 0      # H > 16
    assert iha.iha_backward_workspace_bytes(B, N, 16, d, 9, 1) == 0      # H*P > 128
    assert iha.iha_backward_workspace_bytes(B, N, H, d, P, 0) == 0       # fp32
    ins = [fake] * 8
    outs = [fake] * 8

    def call(**kw):
        a = dict(B=B, N=N, H=H, d=d, P=P, mode=1, window=0, dO=fake, dtype=1, ws=None, wsb=0, outs=outs)
        a.update(kw)
        return iha.iha_backward(*ins, a["B"], a["N"], a["H"], a["d"], a["P"], a["mode"], a["window"], a["dO"],
                                *a["outs"], a["dtype"], None, a["ws"], a["wsb"])
    assert call(dO=None) == iha.IHA_ERR_INVALID_ARG
    assert call(outs=[fake] * 7 + [None]) == iha.IHA_ERR_INVALID_ARG
    assert call(mode=2, window=0) == iha.IHA_ERR_INVALID_ARG
    assert call(dtype=0) == iha.IHA_ERR_UNSUPPORTED
    assert call(H=20) == iha.IHA_ERR_UNSUPPORTED
    assert call(dO=fake + 8) == iha.IHA_ERR_INVALID_ARG                 # dO is read by TMA: 16-byte aligned
    assert call(ws=fake, wsb=256) == iha.IHA_ERR_WORKSPACE


def test_register_contracts_hold_in_this_build(iha):
    """The setmaxnreg kernels were compiled to the register count their split assumes
    (the build already refuses otherwise; this reads the same ptxas reports)."""
    import __graft_entry__
    b = __graft_entry__._build_module()
    b.check_register_contracts()
    for frag, (src, const) in b.REG_CONTRACTS.items():
        log = open(os.path.join(b.BUILD, src[:-3] + ".ptxas.txt")).read()
        regs = {k: v for k, v in b._kernel_registers(log).items() if frag in k}
        assert regs and set(regs.values()) == {b._declared_regs(src, const)}


def test_register_contract_check_rejects_a_mismatch(tmp_path, monkeypatch):
    """A kernel compiled to another register count makes the build fail, naming it."""
    import __graft_entry__
    b = __graft_entry__._build_module()
    (tmp_path / "k_fake.ptxas.txt").write_text(
        "ptxas info    : Compiling entry function '_ZN3iha7fake_wsEv' for 'sm_103a'\n"
        "ptxas info    : Used 128 registers, used 16 barriers\n")
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "k_fake.cu").write_text("constexpr int FAKE_LAUNCH_REGS = 168;\n")
    monkeypatch.setattr(b, "BUILD", str(tmp_path))
    monkeypatch.setattr(b, "CSRC", str(csrc))
    monkeypatch.setattr(b, "REG_CONTRACTS", {"fake_ws": ("k_fake.cu", "FAKE_LAUNCH_REGS")})
    with pytest.raises(RuntimeError, match="_ZN3iha7fake_wsEv: 128 registers"):
        b.check_register_contracts()
    (tmp_path / "k_fake.ptxas.txt").write_text(
        "ptxas info    : Compiling entry function '_ZN3iha7fake_wsEv' for 'sm_103a'\n"
        "ptxas info    : Used 168 registers, used 16 barriers\n")
    b.check_register_contracts()
