"""The allocation-free projection entry point against the workspace-based one.

Some callers cannot allocate device memory at all (an engine that owns every byte and
forbids allocation while it executes, or a latency-critical loop where cudaMalloc would
synchronise the device). evs_projection_noalloc serves them with scratch compiled into the
library. This test calls it twice in a row through the C-ABI and checks both results
against evs_debug_projection on the same inputs, and against an fp32 matmul of the same
bf16 operands, at the projection tests' tolerance: over the whole output and also per
token row and per 128-channel tile, so that one wrong row or tile cannot hide in the
norm. It reads the array's flag word (zero after correct calls, cleared on read), checks
that a shape whose partial sums would not fit at the default split runs with fewer splits,
and that a width beyond the array's counters is rejected. It lives in its own file,
collected last, and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def ver():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from lossless_speculative_verify_gb300.build import build
    build()
    from lossless_speculative_verify_gb300 import DeviceWeights, Verifier, make_config
    from synth import LayerSpec, gen_weights, get_workload
    wl = get_workload("d4096_l32_p8k_bf16").replace(
        layers=(LayerSpec("fir", 3),), batch=4, prefill_chunk=128)
    layers = [(s.kind, s.param) for s in wl.layers]
    cfg = make_config(wl.d, layers, wl.head_dim, wl.gamma, wl.batch, wl.n_cand, 1024,
                      wl.prefill_chunk, "bf16", "greedy")
    return Verifier(cfg, DeviceWeights(layers, gen_weights(wl), "bf16"))


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _flags(lib, clear):
    f = ctypes.c_uint32(0xFFFFFFFF)
    assert lib.evs_projection_noalloc_flags(ctypes.byref(f), clear, _stream()) == 0
    return f.value


def _assert_close(Y, ref, what):
    """Whole-output relative L2 error, and the worst over token rows and over 128-channel
    tiles (each relative to the same slice of the reference)."""
    err = ((Y - ref).norm() / ref.norm()).item()
    assert err < TOL, f"{what}: rel err {err:.2e}"
    rows = ((Y - ref).norm(dim=1) / ref.norm(dim=1).clamp_min(1e-30)).max().item()
    assert rows < TOL, f"{what}: worst row rel err {rows:.2e}"
    M, N = ref.shape
    d = (Y - ref).reshape(M, N // 128, 128).permute(1, 0, 2).reshape(N // 128, -1)
    r = ref.reshape(M, N // 128, 128).permute(1, 0, 2).reshape(N // 128, -1)
    tiles = (d.norm(dim=1) / r.norm(dim=1).clamp_min(1e-30)).max().item()
    assert tiles < TOL, f"{what}: worst channel tile rel err {tiles:.2e}"


def _check(ver, M, N, K, accumulate, seed):
    lib = ver.lib
    g = torch.Generator(device="cuda").manual_seed(seed)
    X = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    base = torch.randn(M, N, device="cuda", generator=g)
    ref = base.clone()
    assert lib.evs_debug_projection(ver.h, _vp(X), M, _vp(W), _vp(ref), M, N, K, N, accumulate) == 0
    mm = X.float() @ W.float().t() + (base if accumulate else 0)
    for call in range(2):                    # two calls in a row share the static scratch
        Y = base.clone()
        assert lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, N, K, N, accumulate,
                                          _stream()) == 0
        torch.cuda.synchronize()
        _assert_close(Y, ref, f"call {call} vs workspace projection")
        _assert_close(Y, mm, f"call {call} vs fp32 matmul")


@pytest.mark.parametrize("M,N,K", [(13, 1024, 1024), (52, 3072, 1024), (208, 512, 1024), (7, 512, 1024),
                                   (300, 128, 64), (13, 512, 4096), (52, 512, 4096)])
@pytest.mark.parametrize("accumulate", [0, 1])
def test_noalloc_matches_workspace_projection(ver, M, N, K, accumulate):
    _check(ver, M, N, K, accumulate, M + N + K + accumulate)
    assert _flags(ver.lib, clear=1) == 0     # no bounded wait gave up
    assert _flags(ver.lib, clear=0) == 0     # and the word reads zero after the clear


def test_noalloc_caps_splits_to_the_array(ver):
    """512 x 1024 at K=4096 splits 8 ways by default (8 x 512 x 1024 partial floats, more than
    the 2^21 the array holds); here it runs with fewer splits and gives the same result."""
    _check(ver, 512, 1024, 4096, 0, 11)
    assert _flags(ver.lib, clear=1) == 0


def test_noalloc_rejects_width_beyond_counters(ver):
    M, K, N = 1, 64, 32768 + 128             # one 128-channel tile more than the counters cover
    X = torch.zeros(M, K, device="cuda", dtype=torch.bfloat16)
    W = torch.zeros(N, K, device="cuda", dtype=torch.bfloat16)
    Y = torch.zeros(M, N, device="cuda")
    lib = ver.lib
    assert lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, N, K, N, 0, _stream()) == 2
    assert lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, 100, K, N, 0, _stream()) == 1
    assert lib.evs_projection_noalloc_flags(None, 0, _stream()) == 1
