"""The allocation-free projection entry point against the workspace-based one.

Some callers cannot allocate device memory at all (an engine that owns every byte and
forbids allocation while it executes, or a latency-critical loop where cudaMalloc would
synchronise the device). evs_projection_noalloc serves them with scratch compiled into the
library. This test calls it twice in a row through the C-ABI and checks both results
against evs_debug_projection on the same inputs, at the projection tests' tolerance, and
that a shape whose split-K scratch does not fit is rejected. It lives in its own file,
collected last, and passes both alone in a fresh process and after the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("M,N,K", [(13, 1024, 1024), (52, 3072, 1024), (208, 512, 1024), (7, 512, 1024),
                                   (300, 128, 64), (13, 512, 4096), (52, 512, 4096)])
@pytest.mark.parametrize("accumulate", [0, 1])
def test_noalloc_matches_workspace_projection(ver, M, N, K, accumulate):
    lib = ver.lib
    g = torch.Generator(device="cuda").manual_seed(M + N + K + accumulate)
    X = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    base = torch.randn(M, N, device="cuda", generator=g)
    ref = base.clone()
    assert lib.evs_debug_projection(ver.h, _vp(X), M, _vp(W), _vp(ref), M, N, K, N, accumulate) == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                       # two calls in a row share the static scratch
        Y = base.clone()
        assert lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, N, K, N, accumulate,
                                          stream) == 0
        torch.cuda.synchronize()
        err = (Y - ref).norm() / ref.norm()
        assert err < 1e-5, f"rel err {err:.2e}"


def test_noalloc_rejects_scratch_overflow(ver):
    M, N, K = 512, 1024, 4096                # 8 splits x 512 x 1024 partial floats > 2^21
    X = torch.zeros(M, K, device="cuda", dtype=torch.bfloat16)
    W = torch.zeros(N, K, device="cuda", dtype=torch.bfloat16)
    Y = torch.zeros(M, N, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert ver.lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, N, K, N, 0, stream) == 2
    assert ver.lib.evs_projection_noalloc(_vp(X), M, _vp(W), _vp(Y), M, 100, K, N, 0, stream) == 1
