"""The tcgen05 projection kernel against a plain fp32 PyTorch matmul of the same bf16
operands: shapes span one and several 128-channel tiles, split-K and single-split grids,
token counts from 1 to 512 (ragged, exactly 16/256, and the two-accumulator case), plain
stores and residual accumulation, and repeated launches (split-K counters reset)."""
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
    wl = get_workload("d1024_l8_p8k_bf16").replace(
        layers=(LayerSpec("fir", 3), LayerSpec("attn", 8)), batch=4, prefill_chunk=128)
    cfg = make_config(wl.d, [(s.kind, s.param) for s in wl.layers], wl.head_dim, wl.gamma, wl.batch,
                      wl.n_cand, 1024, wl.prefill_chunk, "bf16", "greedy")
    return Verifier(cfg, DeviceWeights([(s.kind, s.param) for s in wl.layers], gen_weights(wl), "bf16"))


def _proj(ver, X, W, Y, accumulate):
    M, K = X.shape
    N = W.shape[0]
    st = ver.lib.evs_debug_projection(ver.h, ctypes.c_void_p(X.data_ptr()), X.shape[0],
                                      ctypes.c_void_p(W.data_ptr()), ctypes.c_void_p(Y.data_ptr()),
                                      M, N, K, Y.shape[1], accumulate)
    assert st == 0


@pytest.mark.parametrize("M", [1, 7, 13, 16, 17, 52, 208, 256, 300, 512])
@pytest.mark.parametrize("N,K", [(128, 64), (1024, 1024), (3072, 1024), (512, 1024)])
def test_projection_matches_fp32_matmul(ver, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7919 + N + K)
    X = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    ref = X.float() @ W.float().t()
    for accumulate in (0, 1):
        base = torch.randn(M, N, device="cuda", generator=g)
        Y = base.clone()
        for _ in range(2):                       # second launch reuses the split-K counters
            if accumulate:
                Y.copy_(base)
            _proj(ver, X, W, Y, accumulate)
            torch.cuda.synchronize()
            want = ref + base if accumulate else ref
            err = (Y - want).norm() / want.norm()
            assert err < 1e-5, f"M={M} N={N} K={K} acc={accumulate}: rel err {err:.2e}"
    assert ver.flags() == 0


@pytest.fixture(scope="module")
def ver4096():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from lossless_speculative_verify_gb300.build import build
    build()
    from lossless_speculative_verify_gb300 import DeviceWeights, Verifier, make_config
    from synth import LayerSpec, gen_weights, get_workload
    wl = get_workload("d4096_l8_p32k_b4c4_bf16").replace(layers=(LayerSpec("fir", 3),))
    layers = [(s.kind, s.param) for s in wl.layers]
    cfg = make_config(wl.d, layers, 128, wl.gamma, wl.batch, wl.n_cand, 1024, wl.prefill_chunk, "bf16",
                      "sampling")
    return Verifier(cfg, DeviceWeights(layers, gen_weights(wl), "bf16"))


@pytest.mark.parametrize("M", [13, 52, 208, 256])
@pytest.mark.parametrize("N", [512, 4096, 12288])
def test_projection_width_4096(ver4096, M, N):
    """The decode shapes of the 4096-wide workloads (split-K through a cluster or the
    global scratch, and unsplit)."""
    K = 4096
    g = torch.Generator(device="cuda").manual_seed(M * 31 + N)
    X = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
    ref = X.float() @ W.float().t()
    Y = torch.zeros(M, N, device="cuda")
    for _ in range(2):
        _proj(ver4096, X, W, Y, 0)
        torch.cuda.synchronize()
        err = (Y - ref).norm() / ref.norm()
        assert err < 1e-5, f"M={M} N={N}: rel err {err:.2e}"
    assert ver4096.flags() == 0
