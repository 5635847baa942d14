"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (written here, derived in the design notes):
  float32 path:  max|err| <= 1e-4 * max|O|
  bfloat16 path: RMS(err) <= 2e-2 * RMS(O) over the compared rows, and every
                 compared row within 0.1 of its own RMS (a structural error --
                 a wrong index, mask or scale -- gives O(1) per-row errors,
                 while bf16 rounding of Qbar/Kbar/Vbar, P and the output gives
                 about 1e-2 at most).
Small problems compare every output element; the five full-size workloads
compare sampled rows (first/last tokens, tile and window edges) of the very
launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import iha_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

BF16_RMS_TOL = 2e-2
BF16_ROW_TOL = 0.1
F32_MAX_TOL = 1e-4


@pytest.fixture(scope="module")
def iha():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_variant_gb300 as m
    return m


def to_dev(inp):
    return {k: v.to("cuda:0").contiguous() for k, v in inp.items()}


def run_gpu(iha, w, inp=None, dinp=None):
    if dinp is None:
        dinp = to_dev(inp)
    out = iha.forward(dinp, H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window)
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    return out


def oracle_rows(w, inp, rows=None, projection="c"):
    f = gi.as_f64(inp)
    return oracle.forward(f["X"], f["W_Q"], f["W_K"], f["W_V"], f["alpha_Q"], f["alpha_K"], f["alpha_V"],
                          f["R"], H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window, rows=rows,
                          projection=projection)


def rms(a):
    return float(np.sqrt(np.mean(np.square(a))))


def assert_parity(w, got, ref):
    got = np.asarray(got, dtype=np.float64).reshape(-1, w.D)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, w.D)
    assert np.isfinite(got).all()
    err = got - ref
    if w.dtype == "f32":
        e = float(np.max(np.abs(err)) / np.max(np.abs(ref)))
        assert e <= F32_MAX_TOL, f"{w.name}: max|err|/max|O| = {e:.3e}"
        return e
    e = rms(err) / rms(ref)
    row = np.sqrt(np.mean(err ** 2, axis=1)) / np.maximum(np.sqrt(np.mean(ref ** 2, axis=1)), 1e-30)
    assert e <= BF16_RMS_TOL, f"{w.name}: RMS(err)/RMS(O) = {e:.3e}"
    assert row.max() <= BF16_ROW_TOL, f"{w.name}: worst row error {row.max():.3e} at row {int(row.argmax())}"
    return e


# ---------------------------------------------------------------------------
# every element, against the oracle
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_f32_nomask", "bf16_causal_n1024"])
def test_small_workloads_every_element(iha, name):
    w = gi.WORKLOADS[name]
    inp = gi.make_inputs(w)
    got = run_gpu(iha, w, inp).double().cpu().numpy()
    assert_parity(w, got, oracle_rows(w, inp))


W = gi.Workload
C, NM, WN = gi.MASK_CAUSAL, gi.MASK_NONE, gi.MASK_WINDOW
EDGE = [
    W("n1_p1", B=1, N=1, H=2, d=64, P=1, mask_mode=C, window=0, dtype="bf16", seed=21),
    W("n1_p4_nomask", B=2, N=1, H=2, d=128, P=4, mask_mode=NM, window=0, dtype="bf16", seed=22),
    W("n3_nomask", B=1, N=3, H=2, d=64, P=2, mask_mode=NM, window=0, dtype="bf16", seed=23),
    W("one_tile", B=1, N=64, H=2, d=64, P=2, mask_mode=C, window=0, dtype="bf16", seed=24),
    W("ragged_window_D192", B=2, N=100, H=3, d=64, P=2, mask_mode=WN, window=7, dtype="bf16", seed=25),
    W("ragged_p3", B=1, N=333, H=2, d=128, P=3, mask_mode=C, window=0, dtype="bf16", seed=26),
    W("l129_nomask", B=1, N=129, H=2, d=64, P=1, mask_mode=NM, window=0, dtype="bf16", seed=27),
    W("window1_p4", B=1, N=300, H=2, d=128, P=4, mask_mode=WN, window=1, dtype="bf16", seed=28),
    W("window_ge_n", B=1, N=257, H=2, d=64, P=2, mask_mode=WN, window=1000, dtype="bf16", seed=29),
    W("h1_narrow_gemm", B=3, N=130, H=1, d=64, P=1, mask_mode=C, window=0, dtype="bf16", seed=30),
    W("multi_tile_window", B=1, N=1000, H=2, d=128, P=2, mask_mode=WN, window=300, dtype="bf16", seed=31),
    W("p4_causal_d64", B=2, N=200, H=4, d=64, P=4, mask_mode=C, window=0, dtype="bf16", seed=32),
    # tile shapes of the mixing and contraction kernels: H*P = 128 (one token group per
    # tile), 65..127 (padded K, one group, P not dividing 128), 64 with d = 64, H > 16 (folded
    # route, row-mixing contraction; H = 20, d = 128 is the pages' model shape), ragged tokens
    W("hp128_p8", B=1, N=160, H=16, d=128, P=8, mask_mode=C, window=0, dtype="bf16", seed=36),
    W("hp80_p5_window", B=2, N=77, H=16, d=64, P=5, mask_mode=WN, window=9, dtype="bf16", seed=37),
    W("h20_folded", B=1, N=96, H=20, d=128, P=2, mask_mode=C, window=0, dtype="bf16", seed=38),
    W("h16_d64_p4", B=1, N=300, H=16, d=64, P=4, mask_mode=C, window=0, dtype="bf16", seed=39),
    W("h12_ragged_window", B=3, N=111, H=12, d=128, P=2, mask_mode=WN, window=50, dtype="bf16", seed=40),
    W("f32_odd_d", B=2, N=37, H=3, d=17, P=3, mask_mode=C, window=0, dtype="f32", seed=33),
    W("f32_window", B=1, N=50, H=2, d=40, P=2, mask_mode=WN, window=4, dtype="f32", seed=34),
    W("f32_n1", B=1, N=1, H=1, d=8, P=1, mask_mode=NM, window=0, dtype="f32", seed=35),
]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_shapes_every_element(iha, w):
    inp = gi.make_inputs(w)
    got = run_gpu(iha, w, inp).double().cpu().numpy()
    assert_parity(w, got, oracle_rows(w, inp))


# ---------------------------------------------------------------------------
# full-size workloads: sampled rows
# ---------------------------------------------------------------------------

def sample_rows(w, seed=0):
    """Flat output rows (b*N + t) to compare at full size: fixed edge tokens (first and
    last tokens, tile and window edges) of the first and last batch element, plus one
    random token of every 128-row stacked query tile (128/P tokens) of EVERY batch
    element, so that each attention work item of every head has rows under test."""
    toks = {0, 1, 2, 63, 64, 127, 128, 129, 255, 256, w.N // 2, w.N // 2 + 1, w.N - 2, w.N - 1}
    if w.mask_mode == WN:
        toks |= {w.window - 1, w.window, w.window + 1, 2 * w.window}
    toks = {t for t in toks if 0 <= t < w.N}
    rng = np.random.default_rng(1000 + seed)
    per_tile = max(1, 128 // w.P)   # tokens per 128-row stacked tile
    rows = set()
    for b in range(w.B):
        tile_toks = {int(t0 + rng.integers(0, min(per_tile, w.N - t0))) for t0 in range(0, w.N, per_tile)}
        edge = toks if b in (0, w.B - 1) else set()
        rows |= {b * w.N + t for t in tile_toks | edge}
    return sorted(rows)


def one_hot_contraction(H, P, k):
    """R [H][H*P] picking pseudo-block j = (h + k) mod P of head h itself: output head h is
    then exactly that pseudo-head's attention output (no other pseudo-head mixed in), and
    over k = 0..P-1 every (h, j) is picked once."""
    R = torch.zeros(H, H * P, dtype=torch.float32)
    for h in range(H):
        R[h, h * P + (h + k) % P] = 1.0
    return R


FULL = ["bf16_window1024_n4096", "bf16_causal_p4_n8192", "bf16_window4096_n16384"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(iha, name):
    """The launch configuration the benchmark times: one token of every stacked query
    tile of every batch element against the oracle, and a second call bit-identical."""
    w = gi.WORKLOADS[name]
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    out = run_gpu(iha, w, dinp=dinp)
    again = run_gpu(iha, w, dinp=dinp)
    assert torch.equal(out, again), f"{name}: two calls on the same inputs differ"
    got = out.double().cpu().numpy().reshape(w.B * w.N, w.D)
    rows = sample_rows(w)
    ref = oracle_rows(w, inp, rows=rows, projection="numpy")
    assert_parity(w, got[rows], ref)
    # properties that hold at every row
    assert np.isfinite(got).all()


@pytest.mark.parametrize("name", FULL)
def test_full_size_single_pseudo_head_outputs(iha, name):
    """R picks one pseudo-block per head (one_hot_contraction), so every compared output
    element is one attention output element of one pseudo-head, undiluted by the
    contraction over H*P pseudo-heads; run for k = 0..P-1, each (h, j) of every sampled
    tile is compared once."""
    w = gi.WORKLOADS[name]
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    for k in range(w.P):
        R = one_hot_contraction(w.H, w.P, k)
        inp["R"] = R
        dinp["R"] = R.to("cuda:0")
        got = run_gpu(iha, w, dinp=dinp).double().cpu().numpy().reshape(w.B * w.N, w.D)
        rows = sample_rows(w, seed=k + 1)
        ref = oracle_rows(w, inp, rows=rows, projection="numpy")
        assert_parity(w, got[rows], ref)


def test_full_size_mha_special_case(iha):
    """Long-context shape with P = 1, alpha = identity, R = identity: IHA must be
    plain MHA (Definition 1).  Early rows against the independent MHA loop, all
    sampled rows against the IHA oracle (equal to MHA by the inclusion pin)."""
    w = gi.WORKLOADS["bf16_window4096_n16384"].with_(P=1, window=4096, name="mha_case")
    inp = gi.make_inputs(w)
    inp["alpha_Q"] = inp["alpha_K"] = inp["alpha_V"] = gi.identity_mixing(w.H, 1)
    inp["R"] = gi.first_block_contraction(w.H, 1)
    got = run_gpu(iha, w, inp).double().cpu().numpy().reshape(w.N, w.D)
    early = [0, 1, 100, 255]
    f = gi.as_f64(inp)
    ref_mha = oracle.mha(f["X"], f["W_Q"], f["W_K"], f["W_V"], H=w.H, d=w.d, mask_mode=w.mask_mode,
                         window=w.window, rows=early)
    assert_parity(w, got[early], ref_mha)
    rows = sample_rows(w)
    assert_parity(w, got[rows], oracle_rows(w, inp, rows=rows, projection="numpy"))


# ---------------------------------------------------------------------------
# invariants on the GPU
# ---------------------------------------------------------------------------

def test_prefix_isolation_and_determinism(iha):
    """Causal: changing tokens after t0 leaves outputs at t <= t0 bit-identical;
    the same inputs give bit-identical outputs twice."""
    w = W("prefix", B=1, N=700, H=4, d=128, P=2, mask_mode=C, window=0, dtype="bf16", seed=40)
    inp = gi.make_inputs(w)
    a = run_gpu(iha, w, inp)
    a2 = run_gpu(iha, w, inp)
    assert torch.equal(a, a2)
    t0 = 300
    inp2 = dict(inp)
    X2 = inp["X"].clone()
    X2[:, t0 + 1:] = -X2[:, t0 + 1:] * 2
    inp2["X"] = X2
    b = run_gpu(iha, w, inp2)
    assert torch.equal(a[:, :t0 + 1], b[:, :t0 + 1])
    assert not torch.equal(a[:, t0 + 1:], b[:, t0 + 1:])


def test_window_at_least_n_equals_causal(iha):
    w = W("wgen", B=2, N=300, H=2, d=64, P=2, mask_mode=C, window=0, dtype="bf16", seed=41)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    a = run_gpu(iha, w, dinp=dinp)
    b = run_gpu(iha, w.with_(mask_mode=WN, window=w.N), dinp=dinp)
    assert torch.equal(a, b)


def test_repeated_tokens_gpu(iha):
    """All tokens equal: every output row equals the oracle's row (the
    repeated-token closed form is pinned on the oracle side)."""
    w = W("repeat", B=1, N=400, H=4, d=64, P=2, mask_mode=WN, window=50, dtype="bf16", seed=42)
    inp = gi.make_inputs(w)
    inp["X"] = inp["X"][:, :1].repeat(1, w.N, 1).contiguous()
    got = run_gpu(iha, w, inp).double().cpu().numpy()
    assert_parity(w, got, oracle_rows(w, inp))


# ---------------------------------------------------------------------------
# the other entry points give the same bits as iha_forward_ex
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 3])
def test_step_entry_points_match_forward(iha, P):
    """Every way of computing steps 1+2 (fold alpha into W; project the heads, then mix; the
    projection with the mixing in its epilogue) matches the oracle; the route iha_forward_ex
    takes gives its bits exactly."""
    w = W("steps", B=2, N=260, H=4, d=64, P=P, mask_mode=WN, window=40, dtype="bf16", seed=43)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    ref = run_gpu(iha, w, dinp=dinp)
    dt = iha.IHA_DTYPE_BF16
    route = iha.iha_projection_route(w.H, w.d, w.P, dt)
    assert route == 1
    s = torch.cuda.current_stream()
    ora = oracle_rows(w, inp)
    for r in (0, 1, 2):
        QKV = torch.empty(3, w.B, w.H, w.N * w.P, w.d, dtype=torch.bfloat16, device="cuda:0")
        Pbar = torch.empty(w.B, w.N, w.H, w.P, w.d, dtype=torch.bfloat16, device="cuda:0")
        out = torch.empty_like(ref)
        if r == 0:
            Wt = torch.empty(3 * w.H * w.P * w.d, w.D, dtype=torch.bfloat16, device="cuda:0")
            iha.check(iha.iha_fold_weights(dinp["W_Q"], dinp["W_K"], dinp["W_V"], dinp["alpha_Q"],
                                           dinp["alpha_K"], dinp["alpha_V"], w.H, w.d, w.P, dt, Wt, s))
            iha.check(iha.iha_project(dinp["X"], Wt, w.B, w.N, w.H, w.d, w.P, dt, QKV, s))
        elif r == 2:
            Wp = torch.empty(iha.iha_sliced_weights_bytes(w.H, w.d, dt), dtype=torch.uint8, device="cuda:0")
            iha.check(iha.iha_slice_weights(dinp["W_Q"], dinp["W_K"], dinp["W_V"], w.H, w.d, dt, Wp, s))
            iha.check(iha.iha_project_mix(dinp["X"], Wp, dinp["alpha_Q"], dinp["alpha_K"], dinp["alpha_V"], w.B, w.N,
                                          w.H, w.d, w.P, dt, QKV, s))
        else:
            Y = torch.empty(w.B * w.N, 3 * w.D, dtype=torch.bfloat16, device="cuda:0")
            iha.check(iha.iha_project_heads(dinp["X"], dinp["W_Q"], dinp["W_K"], dinp["W_V"], w.B, w.N, w.H,
                                            w.d, dt, Y, s))
            iha.check(iha.iha_mix_heads(Y, dinp["alpha_Q"], dinp["alpha_K"], dinp["alpha_V"], w.B, w.N, w.H,
                                        w.d, w.P, dt, QKV, s))
            # the head projections themselves: X W_s^(m), checked in float64 on a slice
            f = gi.as_f64(inp)
            sl = slice(0, 7)
            yref = f["X"].reshape(-1, w.D)[sl] @ f["W_V"]
            ygot = Y[sl, 2 * w.D:3 * w.D].double().cpu().numpy()
            np.testing.assert_allclose(ygot, yref, rtol=2e-2, atol=2e-2 * np.abs(yref).max())
        iha.check(iha.iha_attention(QKV, w.B, w.N, w.H, w.d, w.P, w.mask_mode, w.window, dt, Pbar, s))
        iha.check(iha.iha_contract(Pbar, dinp["R"], w.B, w.N, w.H, w.d, w.P, dt, out, s))
        torch.cuda.synchronize()
        assert_parity(w, out.double().cpu().numpy(), ora)
        if (r == 2 and route == 1) or (r == 0 and route == 0):
            assert torch.equal(out, ref)
        if r == 0:
            # the folded weights are the mixing sum (checked in float64 on a slice)
            f = gi.as_f64(inp)
            h, j, c = 1, P - 1, 5
            col = sum(f["alpha_K"][m, h, j] * f["W_K"][:, m * w.d + c] for m in range(w.H))
            row = Wt[1 * w.H * w.P * w.d + h * w.P * w.d + j * w.d + c].double().cpu().numpy()
            np.testing.assert_allclose(row, col, rtol=1e-2, atol=1e-2 * np.abs(col).max())


@pytest.mark.parametrize("B,N,H,d,P", [
    (1, 200, 16, 128, 4),   # 16-column slices (32-byte swizzle), the workloads' head count
    (2, 130, 16, 64, 2),    # ragged last token tile
    (1, 77, 8, 128, 2),     # 32-column slices (64-byte swizzle)
    (1, 300, 5, 64, 3),     # N = 160, H*P = 15 (not a multiple of 4)
    (2, 65, 3, 128, 3),     # 64-column slices (128-byte swizzle), N = 192
    (1, 40, 1, 64, 4),      # one head
    (1, 1, 4, 128, 2),      # a single token
    # whole 32-token groups: results leave through shared-memory staging and TMA stores
    (1, 256, 16, 128, 4), (2, 96, 16, 64, 2), (1, 64, 8, 128, 2), (3, 32, 4, 64, 1), (1, 64, 2, 128, 8)])
def test_project_mix_matches_definition(iha, B, N, H, d, P):
    """iha_project_mix writes S~_{h,j} = sum_m alpha_s[m,h,j] X W_s^(m) (Algorithm 1, the mixing
    step) at stacked row t*P + j of head h, for every element: against the sums in float64,
    within the rounding of the stored type (bf16 Qbar/Kbar, f16 Vbar)."""
    w = W("pm", B=B, N=N, H=H, d=d, P=P, mask_mode=C, window=0, dtype="bf16", seed=46)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    QKV = torch.full((3, B, H, N * P, d), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    dt = iha.IHA_DTYPE_BF16
    Wp = torch.full((iha.iha_sliced_weights_bytes(H, d, dt),), 0xFF, dtype=torch.uint8, device="cuda:0")
    iha.check(iha.iha_slice_weights(dinp["W_Q"], dinp["W_K"], dinp["W_V"], H, d, dt, Wp, None))
    iha.check(iha.iha_project_mix(dinp["X"], Wp, dinp["alpha_Q"], dinp["alpha_K"], dinp["alpha_V"], B, N, H, d, P,
                                  dt, QKV, None))
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    f = gi.as_f64(inp)
    X = f["X"].reshape(B, N, H * d)
    for si, (wn, an) in enumerate((("W_Q", "alpha_Q"), ("W_K", "alpha_K"), ("W_V", "alpha_V"))):
        Yh = (X @ f[wn]).reshape(B, N, H, d)                      # X W_s^(m), head m
        ref = np.einsum("mhj,bnmc->bhnjc", f[an], Yh).reshape(B, H, N * P, d)
        got = QKV[si].view(torch.float16) if si == 2 else QKV[si]
        got = got.double().cpu().numpy()
        assert np.isfinite(got).all(), f"set {si}: unwritten elements"
        err = np.abs(got - ref)
        bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -12 * np.abs(ref).max()
        assert (err <= bound).all(), f"set {si}: worst excess {float((err - bound).max()):.3e}"


def test_caller_workspace_and_default_stream_entry(iha):
    w = W("ws", B=1, N=200, H=2, d=128, P=2, mask_mode=C, window=0, dtype="bf16", seed=44)
    dinp = to_dev(gi.make_inputs(w))
    ref = run_gpu(iha, w, dinp=dinp)
    nbytes = iha.iha_workspace_bytes(w.B, w.N, w.H, w.d, w.P, iha.IHA_DTYPE_BF16)
    # every byte NaN (bf16, f16 and fp32 alike): a read of workspace the call did not write
    # first would reach the output
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda:0")
    out = iha.forward(dinp, H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    out2 = torch.empty_like(ref)
    torch.cuda.synchronize()
    iha.check(iha.iha_forward(dinp["X"], dinp["W_Q"], dinp["W_K"], dinp["W_V"], dinp["alpha_Q"],
                              dinp["alpha_K"], dinp["alpha_V"], dinp["R"], w.B, w.N, w.H, w.d, w.P,
                              w.mask_mode, w.window, out2))
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)


@pytest.mark.parametrize("B,N,H,d,P,mode,window", [
    (2, 150, 2, 64, 2, C, 0),        # unfolded route, attention per batch element
    (3, 130, 2, 128, 4, WN, 40),     # three batch elements: three chunks
    (1, 700, 4, 128, 4, C, 0),       # one sequence: one attention after the last projection chunk
    (1, 520, 2, 64, 2, WN, 100),     # the same under a window
    (1, 300, 2, 64, 2, NM, 0),       # and without a mask
    (1, 777, 4, 128, 3, WN, 60),     # P does not divide 256: one attention, chunks of 194-195 tokens
    (2, 99, 4, 64, 1, C, 0)])        # folded route (P = 1): the plain sequence
def test_forward_host_buffers(iha, B, N, H, d, P, mode, window):
    w = W("host", B=B, N=N, H=H, d=d, P=P, mask_mode=mode, window=window, dtype="bf16", seed=45)
    inp = gi.make_inputs(w)
    ref = run_gpu(iha, w, inp)
    hin = {k: v.contiguous().pin_memory() for k, v in inp.items()}
    out = torch.empty(w.B, w.N, w.D, dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()
    nbytes = iha.iha_host_buffer_bytes(w.B, w.N, w.H, w.d, w.P, iha.IHA_DTYPE_BF16)
    buf = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda:0")   # NaN bytes: nothing read unwritten
    for dev_buf in (None, buf):
        out.zero_()
        rc = iha.iha_forward_host(hin["X"], hin["W_Q"], hin["W_K"], hin["W_V"], hin["alpha_Q"], hin["alpha_K"],
                                  hin["alpha_V"], hin["R"], w.B, w.N, w.H, w.d, w.P, w.mask_mode, w.window, out,
                                  iha.IHA_DTYPE_BF16, s, dev_buf, nbytes if dev_buf is not None else 0)
        iha.check(rc, "iha_forward_host")
        assert torch.equal(out, ref.cpu())


def test_concurrent_streams_match_sequential(iha):
    """Two layers of different shapes and masks run at once on two streams, each with its own
    workspace, 8 times over: every result equals the same call run alone, bit for bit (the
    attention launches draw their work counters from a shared ring)."""
    ws = [W("conc_a", B=2, N=700, H=4, d=128, P=2, mask_mode=C, window=0, dtype="bf16", seed=61),
          W("conc_b", B=1, N=900, H=8, d=64, P=4, mask_mode=WN, window=100, dtype="bf16", seed=62)]
    dins = [to_dev(gi.make_inputs(w)) for w in ws]
    refs = [run_gpu(iha, w, dinp=di) for w, di in zip(ws, dins)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for _ in range(8):
        for w, di, st in zip(ws, dins, streams):
            nb = iha.iha_workspace_bytes(w.B, w.N, w.H, w.d, w.P, iha.IHA_DTYPE_BF16)
            buf = torch.empty(nb, dtype=torch.uint8, device="cuda:0")
            with torch.cuda.stream(st):
                outs.append((iha.forward(di, H=w.H, d=w.d, P=w.P, mask_mode=w.mask_mode, window=w.window,
                                         stream=st, workspace=buf), buf))
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    for i, (o, _) in enumerate(outs):
        assert torch.equal(o, refs[i % 2]), i


def test_device_wait_timeout_is_reported(iha):
    """A wait that nothing will satisfy gives up after its limit, records its
    site, and the host reads IHA_ERR_TIMEOUT; the context stays usable."""
    assert iha.iha_check_device_status()[0] == iha.IHA_OK
    iha.check(iha.iha_selftest_wait_timeout(None, 20))
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_ERR_TIMEOUT and code == 0x1000 | 99
    assert iha.iha_check_device_status() == (iha.IHA_OK, 0)
    w = W("after_timeout", B=1, N=64, H=2, d=64, P=2, mask_mode=C, window=0, dtype="bf16", seed=46)
    inp = gi.make_inputs(w)
    assert_parity(w, run_gpu(iha, w, inp).double().cpu().numpy(), oracle_rows(w, inp))


# ---------------------------------------------------------------------------
# layer stack (the hybrid local/global schedule): the stack entry point equals the chain of
# single-layer calls bit for bit, and every layer matches the oracle on its own input
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("P_local,N", [(2, 300), (4, 257)])
def test_layer_stack(iha, P_local, N):
    B, H, d = 2, 4, 64
    layers = gi.make_stack_inputs(B, N, H, d, "bf16", seed=60 + P_local, schedule=gi.local_global_schedule(N, P_local))
    keys = ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")
    dev = [{k: L[k].to("cuda:0").contiguous() for k in keys} for L in layers]
    for dl, L in zip(dev, layers):
        dl.update(P=L["P"], mask_mode=L["mask_mode"], window=L["window"])
    X = layers[0]["X"].to("cuda:0").contiguous()
    out = torch.empty_like(X)
    iha.check(iha.iha_forward_stack(X, dev, B, N, H, d, iha.IHA_DTYPE_BF16, out), "iha_forward_stack")
    torch.cuda.synchronize()
    x = X
    for l, (dl, L) in enumerate(zip(dev, layers)):
        w = L["workload"]
        y = run_gpu(iha, w, dinp=dict({k: dl[k] for k in keys}, X=x))
        inp = {k: L[k] for k in keys}
        inp["X"] = x.cpu()
        assert_parity(w, y.double().cpu().numpy(), oracle_rows(w, inp))
        x = y
    assert torch.equal(out, x)


def test_layer_stack_full_size(iha):
    """The stack the benchmark times (causal P=4 N=8192 layer's shape: four window-256 P=4
    layers, then the global P=1 causal layer): bit for bit the chain of single-layer calls,
    and each layer against the oracle on its own input at the full-size sampled rows."""
    B, N, H, d = 1, 8192, 16, 128
    layers = gi.make_stack_inputs(B, N, H, d, "bf16", seed=80, schedule=gi.local_global_schedule(N, 4))
    keys = ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")
    dev = [{k: L[k].to("cuda:0").contiguous() for k in keys} for L in layers]
    for dl, L in zip(dev, layers):
        dl.update(P=L["P"], mask_mode=L["mask_mode"], window=L["window"])
    X = layers[0]["X"].to("cuda:0").contiguous()
    out = torch.full_like(X, float("nan"))
    iha.check(iha.iha_forward_stack(X, dev, B, N, H, d, iha.IHA_DTYPE_BF16, out), "iha_forward_stack")
    torch.cuda.synchronize()
    x = X
    for dl, L in zip(dev, layers):
        w = L["workload"]
        y = run_gpu(iha, w, dinp=dict({k: dl[k] for k in keys}, X=x))
        inp = {k: L[k] for k in keys}
        inp["X"] = x.cpu()
        rows = sample_rows(w)
        got = y.double().cpu().numpy().reshape(B * N, w.D)
        assert_parity(w, got[rows], oracle_rows(w, inp, rows=rows, projection="numpy"))
        x = y
    assert torch.equal(out, x)


# ---------------------------------------------------------------------------
# incremental decoding: prefill a prompt, then decode token by token; every decoded row
# must be the row the forward pass gives that token of the whole sequence (the oracle)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,d,P,mode,window,T", [
    (4, 64, 2, C, 0, 37), (4, 64, 8, WN, 5, 37), (16, 128, 4, C, 0, 37), (3, 128, 3, WN, 20, 37),
    (2, 128, 1, C, 0, 37),
    # long caches: many 128-row tiles per chunk, several chunks, a ragged last tile, and (window)
    # a first readable row that is not tile-aligned
    (2, 128, 4, C, 0, 700), (3, 128, 2, WN, 333, 900),
    # more than 32 chunks per head (36 one-tile chunks: the chunk merge's second lane half)
    (2, 64, 4, C, 0, 1150),
    # window 1: each decoded token reads only its own P pseudo-keys
    (2, 128, 4, WN, 1, 37), (4, 64, 2, WN, 1, 37)])
def test_decode_matches_oracle(iha, H, d, P, mode, window, T):
    B, steps = 2, 4
    n_all = T + steps
    w = gi.Workload("decode", B=B, N=n_all, H=H, d=d, P=P, mask_mode=mode, window=window, dtype="bf16", seed=70 + P)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    D = w.D
    cap = n_all + 3
    Kc = torch.zeros(B, H, cap * P, d, dtype=torch.bfloat16, device="cuda:0")
    Vc = torch.zeros(B, H, cap * P, d, dtype=torch.float16, device="cuda:0")
    X = dinp["X"]
    wts = [dinp[k] for k in ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")]
    out_prompt = torch.empty(B, T, D, dtype=torch.bfloat16, device="cuda:0")
    iha.check(iha.iha_prefill(X[:, :T].contiguous(), *wts, B, T, H, d, P, mode, window, out_prompt, Kc, Vc, cap,
                              iha.IHA_DTYPE_BF16), "iha_prefill")
    dec = []
    for s in range(steps):
        t = T + s
        o = torch.empty(B, D, dtype=torch.bfloat16, device="cuda:0")
        iha.check(iha.iha_decode_step(X[:, t].contiguous(), *wts, B, H, d, P, mode, window, Kc, Vc, cap, t, o,
                                      iha.IHA_DTYPE_BF16), "iha_decode_step")
        dec.append(o)
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    rows = [b * n_all + t for b in range(B) for t in range(T, n_all)]
    got = torch.stack(dec, 1).reshape(B * steps, D).double().cpu().numpy()    # [b][step] = rows order
    assert_parity(w, got, oracle_rows(w, inp, rows=rows))
    # the prompt's rows come from the forward pass (rows of a prefix do not depend on later tokens)
    rows_p = [b * n_all + t for b in range(B) for t in range(T)]
    assert_parity(w, out_prompt.reshape(B * T, D).double().cpu().numpy(), oracle_rows(w, inp, rows=rows_p))


@pytest.mark.parametrize("name", FULL)
def test_decode_full_size_last_token(iha, name):
    """The full-size workloads as `bench.py --decode` runs them: prefill N-1 tokens, then
    decode token N-1 over the whole cache; its row against the oracle's row of the forward
    over the whole sequence, and sampled prefill rows likewise."""
    w = gi.WORKLOADS[name]
    B, N, H, d, P, D = w.B, w.N, w.H, w.d, w.P, w.D
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    wts = [dinp[k] for k in ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")]
    Kc = torch.zeros(B, H, N * P, d, dtype=torch.bfloat16, device="cuda:0")
    Vc = torch.zeros(B, H, N * P, d, dtype=torch.float16, device="cuda:0")
    X = dinp["X"]
    out_prompt = torch.empty(B, N - 1, D, dtype=torch.bfloat16, device="cuda:0")
    iha.check(iha.iha_prefill(X[:, :N - 1].contiguous(), *wts, B, N - 1, H, d, P, w.mask_mode, w.window, out_prompt,
                              Kc, Vc, N, iha.IHA_DTYPE_BF16), "iha_prefill")
    o = torch.empty(B, D, dtype=torch.bfloat16, device="cuda:0")
    iha.check(iha.iha_decode_step(X[:, N - 1].contiguous(), *wts, B, H, d, P, w.mask_mode, w.window, Kc, Vc, N,
                                  N - 1, o, iha.IHA_DTYPE_BF16), "iha_decode_step")
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    rows = [b * N + N - 1 for b in range(B)]
    assert_parity(w, o.double().cpu().numpy(), oracle_rows(w, inp, rows=rows, projection="numpy"))
    prows = [r for r in sample_rows(w) if r % N < N - 1]
    got_p = out_prompt.double().cpu().numpy().reshape(B, N - 1, D)
    assert_parity(w, np.stack([got_p[r // N, r % N] for r in prows]),
                  oracle_rows(w, inp, rows=prows, projection="numpy"))


@pytest.mark.parametrize("d,P", [(64, 2), (128, 4)])
def test_decode_from_empty_cache(iha, d, P):
    """t = 0: the token reads only its own P pseudo-keys."""
    B, H = 3, 4
    w = gi.Workload("decode0", B=B, N=1, H=H, d=d, P=P, mask_mode=C, window=0, dtype="bf16", seed=77)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    wts = [dinp[k] for k in ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")]
    Kc = torch.zeros(B, H, 2 * P, d, dtype=torch.bfloat16, device="cuda:0")
    Vc = torch.zeros(B, H, 2 * P, d, dtype=torch.float16, device="cuda:0")
    o = torch.empty(B, w.D, dtype=torch.bfloat16, device="cuda:0")
    iha.check(iha.iha_decode_step(dinp["X"][:, 0].contiguous(), *wts, B, H, d, P, C, 0, Kc, Vc, 2, 0, o,
                                  iha.IHA_DTYPE_BF16))
    torch.cuda.synchronize()
    assert_parity(w, o.double().cpu().numpy(), oracle_rows(w, inp))


@pytest.mark.parametrize("d,P,fill", [(128, 4, "nan"), (64, 2, "inf"), (128, 2, "nan")])
def test_decode_ignores_unwritten_cache_rows(iha, d, P, fill):
    """Cache rows past the current token may hold any bits (a cache allocated without
    initialisation): NaN or Inf there, read by the last tile of a chunk and masked out,
    must not reach the output; nor may NaN bytes in a caller-provided workspace."""
    B, H, T, steps = 2, 2, 300, 2
    n_all = T + steps
    w = gi.Workload("decode_fill", B=B, N=n_all, H=H, d=d, P=P, mask_mode=C, window=0, dtype="bf16", seed=81)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    wts = [dinp[k] for k in ("W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")]
    cap = n_all + 40
    Kc = torch.full((B, H, cap * P, d), float(fill), dtype=torch.bfloat16, device="cuda:0")
    Vc = torch.full((B, H, cap * P, d), float(fill), dtype=torch.float16, device="cuda:0")
    X = dinp["X"]
    out_prompt = torch.empty(B, T, w.D, dtype=torch.bfloat16, device="cuda:0")
    iha.check(iha.iha_prefill(X[:, :T].contiguous(), *wts, B, T, H, d, P, C, 0, out_prompt, Kc, Vc, cap,
                              iha.IHA_DTYPE_BF16), "iha_prefill")
    # the caller's workspace starts as NaN bytes too: nothing in it may be read before it is written
    nws = iha.iha_decode_workspace_bytes(B, H, d, P)
    ws = torch.full((nws,), 0xFF, dtype=torch.uint8, device="cuda:0")
    dec = []
    for s in range(steps):
        o = torch.full((B, w.D), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        iha.check(iha.iha_decode_step(X[:, T + s].contiguous(), *wts, B, H, d, P, C, 0, Kc, Vc, cap, T + s, o,
                                      iha.IHA_DTYPE_BF16, None, ws, nws), "iha_decode_step")
        dec.append(o)
    torch.cuda.synchronize()
    got = torch.stack(dec, 1).reshape(B * steps, w.D).double().cpu().numpy()
    assert np.isfinite(got).all()
    rows = [b * n_all + t for b in range(B) for t in range(T, n_all)]
    assert_parity(w, got, oracle_rows(w, inp, rows=rows))


# ---------------------------------------------------------------------------
# backward pass: every gradient against the fp64 autograd oracle (oracle/backward.py)
# ---------------------------------------------------------------------------

BWD_TOL = 3e-2   # RMS(err) <= BWD_TOL * RMS(ref) per gradient tensor ...
# ... + CANCEL_TOL * RMS(the gradient reached through the scores by P * D alone): D =
# dPbar . Pbar is formed from the bf16 attention output (relative error ~2^-8), and
# dS = P (dP - D) inherits that error at the size of P * D even where dP - D cancels
CANCEL_TOL = 2.0 ** -6
# ... and, for the four gradients that are sums over all tokens and columns of a product of two
# bf16-stored tensors (dalpha_Q/K/V, dR), + GRAM_TOL * RMS(sqrt(sum of the squared terms)): the
# terms can cancel to a result far below their size, so an error relative to the result alone
# is ill-conditioned there; per-term relative errors of about 2^-8 (bf16 storage of both
# factors) give a sum error of about 2^-8 * sqrt(sum term^2), allowed four times over
GRAM_TOL = 2.0 ** -6


@pytest.mark.parametrize("B,N,H,d,P,mode,window", [
    (2, 40, 4, 64, 2, C, 0), (1, 37, 4, 64, 3, WN, 9), (1, 50, 2, 128, 4, C, 0),
    (2, 33, 4, 64, 1, NM, 0), (1, 45, 16, 64, 2, WN, 20), (1, 70, 8, 128, 2, C, 0),
    # several 128-row tiles and 64-row blocks with a ragged tail: stacked lengths 600, 800, 1024
    (1, 300, 4, 64, 2, WN, 37), (1, 200, 4, 128, 4, WN, 50), (1, 512, 8, 128, 2, C, 0),
    # the causal N=1024 d=64 P=2 workload's shape with one batch element (stacked length 2048)
    (1, 1024, 16, 64, 2, C, 0),
    # degenerate cases: one token; window 1 (each pseudo-query reads its own token's P
    # pseudo-keys); a window >= N (= causal); H*P = 128 with P = 8; one head (D = 64, narrower
    # than one GEMM tile, and one row of the token grams)
    (1, 1, 2, 64, 1, C, 0), (2, 60, 4, 128, 2, WN, 1), (1, 90, 2, 64, 3, WN, 500), (1, 40, 16, 64, 8, C, 0),
    (3, 33, 1, 64, 2, C, 0),
    # the large workloads' heads (H = 16, d = 128, D = 2048: the gradient GEMMs at full width)
    # with P = 4 causal and P = 2 windowed, stacked length 2048 (16 resident tiles per head)
    (1, 512, 16, 128, 4, C, 0), (1, 1024, 16, 128, 2, WN, 256)])
def test_backward_matches_oracle(iha, B, N, H, d, P, mode, window):
    from oracle import backward as bwd
    w = gi.Workload("bwd", B=B, N=N, H=H, d=d, P=P, mask_mode=mode, window=window, dtype="bf16", seed=90 + P)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    D = w.D
    g = torch.Generator().manual_seed(1234 + N)
    dO = torch.randn(B, N, D, generator=g).to(torch.bfloat16)
    # NaN-filled outputs: an element the call leaves unwritten fails the finiteness check
    dev = lambda shape, dt=torch.bfloat16: torch.full(shape, float("nan"), dtype=dt, device="cuda:0")
    out = {"X": dev((B, N, D)), "W_Q": dev((D, D)), "W_K": dev((D, D)), "W_V": dev((D, D)),
           "alpha_Q": dev((H, H, P), torch.float32), "alpha_K": dev((H, H, P), torch.float32),
           "alpha_V": dev((H, H, P), torch.float32), "R": dev((H, H * P), torch.float32)}
    iha.check(iha.iha_backward(*(dinp[k] for k in bwd.PARAMS), B, N, H, d, P, mode, window,
                               dO.to("cuda:0").contiguous(), *(out[k] for k in bwd.PARAMS), iha.IHA_DTYPE_BF16),
              "iha_backward")
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    ref = bwd.backward(gi.as_f64(inp), dO.double(), H=H, d=d, P=P, mask_mode=mode, window=window)
    scale = bwd.cancellation_scale(gi.as_f64(inp), dO.double(), H=H, d=d, P=P, mask_mode=mode, window=window)
    terms = bwd.gram_term_scale(gi.as_f64(inp), dO.double(), H=H, d=d, P=P, mask_mode=mode, window=window)
    for k in bwd.PARAMS:
        got = out[k].double().cpu().numpy()
        r = ref[k].numpy()
        assert np.isfinite(got).all(), k
        err = rms(got - r)
        bound = BWD_TOL * rms(r) + CANCEL_TOL * rms(scale[k].numpy())
        if k in terms:
            bound += GRAM_TOL * rms(terms[k].numpy())
        assert err <= bound, f"{k}: rms err {err:.3g} vs rms ref {rms(r):.3g}, bound {bound:.3g}"


@pytest.mark.parametrize("B,N,H,d,P,mode,window", [
    (2, 150, 4, 64, 2, C, 0), (1, 300, 8, 128, 4, WN, 40), (1, 77, 4, 128, 1, NM, 0),
    # the causal P = 4 workload at full size, as the training benchmark runs it
    (1, 8192, 16, 128, 4, C, 0)])
def test_training_pair_matches_recompute(iha, B, N, H, d, P, mode, window):
    """iha_forward_train + iha_backward_saved give iha_forward's output (the same route at
    every P) and iha_backward's gradients bit for bit."""
    from oracle import backward as bwd
    w = gi.Workload("train", B=B, N=N, H=H, d=d, P=P, mask_mode=mode, window=window, dtype="bf16", seed=31 + P)
    inp = gi.make_inputs(w)
    dinp = to_dev(inp)
    D = w.D
    g = torch.Generator().manual_seed(99 + N)
    dO = torch.randn(B, N, D, generator=g).to(torch.bfloat16).to("cuda:0").contiguous()
    nb = iha.iha_backward_workspace_bytes(B, N, H, d, P, iha.IHA_DTYPE_BF16)
    ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda:0")   # NaN bytes: nothing read unwritten
    out = torch.full((B, N, D), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    args = [dinp[k] for k in bwd.PARAMS] + [B, N, H, d, P, mode, window]
    iha.check(iha.iha_forward_train(*args, out, iha.IHA_DTYPE_BF16, None, ws, nb), "iha_forward_train")

    def grads():   # NaN-filled: an element the calls leave unwritten fails the equality below
        nan = float("nan")
        return {"X": torch.full((B, N, D), nan, dtype=torch.bfloat16, device="cuda:0"),
                **{k: torch.full((D, D), nan, dtype=torch.bfloat16, device="cuda:0") for k in ("W_Q", "W_K", "W_V")},
                **{k: torch.full((H, H, P), nan, dtype=torch.float32, device="cuda:0")
                   for k in ("alpha_Q", "alpha_K", "alpha_V")},
                "R": torch.full((H, H * P), nan, dtype=torch.float32, device="cuda:0")}
    g_saved, g_full = grads(), grads()
    iha.check(iha.iha_backward_saved(*args, dO, *(g_saved[k] for k in bwd.PARAMS), iha.IHA_DTYPE_BF16, None, ws,
                                     nb), "iha_backward_saved")
    iha.check(iha.iha_backward(*args, dO, *(g_full[k] for k in bwd.PARAMS), iha.IHA_DTYPE_BF16), "iha_backward")
    torch.cuda.synchronize()
    rc, code = iha.iha_check_device_status()
    assert rc == iha.IHA_OK, f"device status {rc} word {code:#x}"
    for k in bwd.PARAMS:
        assert torch.equal(g_saved[k], g_full[k]), k
    assert torch.equal(out, run_gpu(iha, w, inp))

