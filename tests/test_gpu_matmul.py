"""GPU tests of the fused decode + product (ndq_matmul_packed) against the
oracle's binary64 reference.

Y[m, n] = sum_k X[m, k] * W[n, k] with W the payload decoded to binary32
(or that decode rounded to bfloat16).  The kernel sums the exact products
(bfloat16 times binary32) with binary32 fused multiply-adds: each term passes through at most K + 13 roundings (its
thread's running sum, 5 warp-shuffle additions, 8 per-warp partials), so
|Y - Y_ref| <= (K + 16) * 2^-24 * sum_k |X W| (the standard recursive
summation bound, doubled for margin below); a bfloat16 output adds one
rounding of at most 2^-8 |Y|.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

import quantized_weight_block_gb300 as ndq  # noqa: E402

DEV = "cuda"
FORMATS = ["gguf:q8_0", "gguf:q4_0", "gguf:iq4_nl", "gguf:q4_k", "gguf:q6_k", "gguf:mxfp4", "gguf:nvfp4", "nvfp4",
           "q4_g64_fp16", "q8_g32_fp16"] + synth.NEXT_FORMATS


def _x_bf16(M, K, seed):
    x = torch.from_numpy(np.random.default_rng(seed).standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
    return x, x.view(torch.int16).numpy().view(np.uint16)


def _run(fmt, N, K, M, w_np, x_t, out_dtype=torch.float32, w_off=0, x_off=0, weights="float32"):
    wbuf = torch.zeros(w_np.size + w_off + 16, dtype=torch.uint8, device=DEV)
    wbuf[w_off:w_off + w_np.size] = torch.from_numpy(w_np).to(DEV)
    w = wbuf[w_off:w_off + w_np.size]
    xbuf = torch.zeros(M * K + x_off + 8, dtype=torch.bfloat16, device=DEV)
    xbuf[x_off:x_off + M * K] = x_t.reshape(-1).to(DEV)
    x = xbuf[x_off:x_off + M * K]
    y = torch.full((M, N), float("nan"), dtype=out_dtype, device=DEV)
    wcode = ndq.NDQ_FLOAT if weights == "float32" else ndq.NDQ_BFLOAT16
    rc = ndq.ndq_matmul_packed(ndq.format_id(fmt), N, K, w.data_ptr(), w_np.size, x.data_ptr(), M, wcode,
                               ndq.out_dtype_code(out_dtype), y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ndq.ndq_status_string(rc)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def _check(got, ref, yabs, K, bf16_out=False, what=""):
    tol = 2.0 * (K + 16) * 2.0 ** -24 * yabs + 1e-30
    if bf16_out:
        tol = tol + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert (err <= tol).all(), f"{what}: worst {np.max(err / tol):.3g} of the bound"


@pytest.fixture(autouse=True)
def _no_device_fault():
    yield
    assert ndq.get_device_fault() == 0


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("weights", ["float32", "bfloat16"])
def test_matmul_against_oracle(orc, fmt, weights):
    N, K, M = 37, 12288, 3  # rows of two segments (8192 + 4096 elements)
    w = synth.payload(fmt, (N, K), seed=11)
    x_t, x_bits = _x_bf16(M, K, 12)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
    _check(_run(fmt, N, K, M, w, x_t, weights=weights), ref, yabs, K, what=f"{fmt} {weights}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("weights", ["float32", "bfloat16"])
def test_matmul_one_row(orc, fmt, weights):
    # one activation row (a generation step): the activations as binary32 in
    # shared memory; rows of two segments (8192 + 4096 elements)
    N, K = 41, 12288
    w = synth.payload(fmt, (N, K), seed=21)
    x_t, x_bits = _x_bf16(1, K, 22)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
    _check(_run(fmt, N, K, 1, w, x_t, weights=weights), ref, yabs, K, what=f"{fmt} M=1 {weights}")


@pytest.mark.parametrize("fmt", ["gguf:q4_k", "gguf:q6_k", "gguf:q8_0", "nvfp4", "fp8_e4m3fn_row_bf16"])
@pytest.mark.parametrize("K,x_off", [(14336, 0), (14336, 1), (20480, 0), (256, 0), (4096, 3)])
def test_matmul_one_row_activation_sources(orc, fmt, K, x_off):
    # one row up to K = 16384 is held in shared memory (converted with
    # 16-byte loads, or element by element when X is not 16-byte aligned);
    # longer rows are read from global memory
    B = synth.GEOMETRY[fmt][0]
    K = K // max(B, 16) * max(B, 16)
    N = 23
    w = synth.payload(fmt, (N, K), seed=K + x_off)
    x_t, x_bits = _x_bf16(1, K, K)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "float32")
    _check(_run(fmt, N, K, 1, w, x_t, x_off=x_off), ref, yabs, K, what=f"{fmt} M=1 K={K} x+{x_off}")


@pytest.mark.parametrize("fmt", ["gguf:q8_0", "gguf:q4_k", "gguf:q6_k", "q8_g32_fp16"])
@pytest.mark.parametrize("N,K", [(1, 512), (300, 4096), (3000, 4096), (77, 8192), (1000, 14336), (5, 16384),
                                 (64, 1536)])
@pytest.mark.parametrize("weights,out", [("float32", torch.float32), ("bfloat16", torch.bfloat16)])
def test_matmul_one_row_lean_kernel(orc, fmt, N, K, weights, out):
    # the lean one-row kernels (K a multiple of 512, aligned rows): X in
    # registers up to K = 4096 and for q8_0 rows too long for the other
    # (one, two or four 16-weight units per lane, 1 to 8 warps per row), X
    # in shared memory above K = 4096 (several iterations per warp); rows
    # wrapping the 3-stage ring (3000 rows), both weight operands and output
    # types
    w = synth.payload(fmt, (N, K), seed=31 + K)
    x_t, x_bits = _x_bf16(1, K, 32)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
    got = _run(fmt, N, K, 1, w, x_t, out_dtype=out, weights=weights)
    _check(got, ref, yabs, K, bf16_out=out == torch.bfloat16, what=f"{fmt} [{N},{K}] {weights} {out}")


@pytest.mark.parametrize("fmt", ["gguf:q8_0", "gguf:q4_k", "gguf:q6_k", "q8_g32_fp16"])
@pytest.mark.parametrize("N,K", [(300, 4096), (4099, 3072), (1000, 512), (77, 1024), (5, 2048), (2000, 2560)])
@pytest.mark.parametrize("M", [2, 3, 5, 8])
@pytest.mark.parametrize("weights,out", [("float32", torch.float32), ("bfloat16", torch.bfloat16)])
def test_matmul_several_rows_lean_kernel(orc, fmt, N, K, M, weights, out):
    # 2..8 activation rows, K a multiple of 512 up to 4096 (the lean kernel
    # for several rows): X padded to 2, 4 or 8 rows, the rows split over
    # warp halves at 8; 1 to 8 iterations per row (5 and 6 leave warps
    # idle), rows wrapping the 3-slot ring with a partial last block (4099)
    w = synth.payload(fmt, (N, K), seed=71 + M)
    x_t, x_bits = _x_bf16(M, K, 72 + M)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
    got = _run(fmt, N, K, M, w, x_t, out_dtype=out, weights=weights)
    _check(got, ref, yabs, K, bf16_out=out == torch.bfloat16, what=f"{fmt} [{N},{K}] M={M} {weights} {out}")


@pytest.mark.parametrize("fmt", ["gguf:q6_k", "gguf:q8_0", "q8_g32_fp16"])
@pytest.mark.parametrize("N,K", [(300, 4608), (77, 256), (1000, 14336), (130, 12288), (4096, 1280)])
@pytest.mark.parametrize("M", [2, 3, 5, 8])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_grouped_tensor_core_exact_weights(orc, fmt, N, K, M, out):
    # gguf:q6_k and q8_0 with binary32 weights and 2..8 activation rows where
    # the lean kernel does not take them (K not a multiple of 512, or above
    # 4096): the tensor core sums codes times X per 16- or 32-weight group
    # into its own TMEM column, the epilogue applies the group scales; row
    # tiles partial, split-K clusters for the short grids (N = 77, 130, 300)
    w = synth.payload(fmt, (N, K), seed=41 + M)
    x_t, x_bits = _x_bf16(M, K, 42 + M)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "float32")
    got = _run(fmt, N, K, M, w, x_t, out_dtype=out)
    _check(got, ref, yabs, K, bf16_out=out == torch.bfloat16, what=f"{fmt} [{N},{K}] M={M} {out}")


@pytest.mark.parametrize("fmt", ["gguf:q6_k", "gguf:q8_0"])
@pytest.mark.parametrize("w_off,M,weights", [(1, 4, "float32"), (6, 3, "float32"), (8, 8, "float32"),
                                             (2, 16, "bfloat16"), (12, 40, "bfloat16")])
def test_tensor_core_products_unaligned_payload(orc, fmt, w_off, M, weights):
    # a payload that starts off a 16-byte boundary: the tensor-core kernels
    # stage its rows by 16-byte lines (no tensor copy) and decode every
    # block at its own byte phase
    N, K = 150, 2048
    w = synth.payload(fmt, (N, K), seed=60 + w_off)
    x_t, x_bits = _x_bf16(M, K, 61)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
    _check(_run(fmt, N, K, M, w, x_t, w_off=w_off, weights=weights), ref, yabs, K,
           what=f"{fmt} +{w_off} M={M} {weights}")


@pytest.mark.parametrize("fmt", ["gguf:q4_k", "gguf:q8_0", "gguf:mxfp4", "gguf:iq3_s", "nvfp4", "fp8_e4m3fn_row_fp16"])
@pytest.mark.parametrize("N,K", [(37, 4096), (13, 2048), (9, 1024), (17, 512), (5, 256), (130, 8192), (3, 12800)])
def test_matmul_whole_rows_per_stage(orc, fmt, N, K):
    # K <= 4096 stages 2..8 whole rows at a time (a partial last unit when N
    # is not a multiple); larger K splits rows into segments
    B = synth.GEOMETRY[fmt][0]
    if K % max(B, 16):
        pytest.skip("K not a multiple of the block")
    w = synth.payload(fmt, (N, K), seed=K + N)
    x_t, x_bits = _x_bf16(2, K, N)
    for weights in ("float32", "bfloat16"):
        ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
        _check(_run(fmt, N, K, 2, w, x_t, weights=weights), ref, yabs, K, what=f"{fmt} {N}x{K} {weights}")


@pytest.mark.parametrize("fmt", ["gguf:q4_k", "gguf:q6_k", "gguf:q8_0", "gguf:iq2_xs", "nvfp4", "fp8_e4m3fn_row_bf16"])
@pytest.mark.parametrize("M", [1, 8, 11])
def test_matmul_rows_of_x_and_bf16_output(orc, fmt, M):
    B = synth.GEOMETRY[fmt][0]
    N, K = 64, 2048 // max(B, 16) * max(B, 16)
    w = synth.payload(fmt, (N, K), seed=M)
    x_t, x_bits = _x_bf16(M, K, 100 + M)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "float32")
    _check(_run(fmt, N, K, M, w, x_t), ref, yabs, K, what=f"{fmt} M={M}")
    _check(_run(fmt, N, K, M, w, x_t, out_dtype=torch.bfloat16), ref, yabs, K, bf16_out=True, what=f"{fmt} M={M} bf16")


@pytest.mark.parametrize("fmt", ["gguf:q4_k", "gguf:q5_0", "gguf:mxfp4", "q6_g64_fp16"])
@pytest.mark.parametrize("w_off,x_off", [(1, 0), (7, 3), (0, 1)])
def test_matmul_unaligned_operands(orc, fmt, w_off, x_off):
    B = synth.GEOMETRY[fmt][0]
    N, K = 19, 3 * 1024 // max(B, 16) * max(B, 16)
    w = synth.payload(fmt, (N, K), seed=w_off)
    x_t, x_bits = _x_bf16(2, K, x_off)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "float32")
    _check(_run(fmt, N, K, 2, w, x_t, w_off=w_off, x_off=x_off), ref, yabs, K, what=f"{fmt} +{w_off}/+{x_off}")


def test_matmul_nvfp4_several_divisors(orc):
    N, K = 12, 64 * 40
    w = synth.payload("nvfp4", (N, K), seed=4, ndiv=4)
    x_t, x_bits = _x_bf16(2, K, 5)
    ref, yabs = orc.matmul_packed("nvfp4", N, K, w, x_bits, "float32")
    _check(_run("nvfp4", N, K, 2, w, x_t), ref, yabs, K, what="nvfp4 D=4")


def test_matmul_is_deterministic():
    fmt, N, K, M = "gguf:q4_k", 256, 4096, 4
    w = synth.payload(fmt, (N, K), seed=1)
    x_t, _ = _x_bf16(M, K, 2)
    a = _run(fmt, N, K, M, w, x_t)
    b = _run(fmt, N, K, M, w, x_t)
    assert np.array_equal(a, b)


def test_matmul_validation_and_empty():
    q4k = ndq.format_id("gguf:q4_k")
    F = ndq.NDQ_FLOAT
    assert ndq.ndq_matmul_packed(q4k, 2, 256, 16, 288, 16, 1, F, ndq.NDQ_FLOAT16, 16) == 9
    assert ndq.ndq_matmul_packed(q4k, 2, 256, 16, 288, 16, 1, ndq.NDQ_FLOAT16, F, 16) == 9
    assert ndq.ndq_matmul_packed(q4k, -1, 256, 16, 0, 16, 1, F, F, 16) == 5
    assert ndq.ndq_matmul_packed(q4k, 2, 100, 16, 0, 16, 1, F, F, 16) == 6
    assert ndq.ndq_matmul_packed(q4k, 2, 256, 16, 287, 16, 1, F, F, 16) == 7
    assert ndq.ndq_matmul_packed(ndq.format_id("fp8_e4m3fn_row_fp16"), 2, 24, 16, 52, 16, 1, F, F, 16) == 6
    assert ndq.ndq_matmul_packed(99, 2, 256, 16, 288, 16, 1, F, F, 16) == 2
    assert ndq.ndq_matmul_packed(q4k, 2, 256, 16, 288, 16, 0, F, F, 0) == 0  # M = 0
    y = torch.full((3, 5), 7.0, dtype=torch.float32, device=DEV)
    assert ndq.ndq_matmul_packed(q4k, 5, 0, 0, 0, 0, 3, F, F, y.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream) == 0  # K = 0: zeros
    torch.cuda.synchronize()
    assert not y.any()


# ---- the tensor-core (tcgen05) path: bfloat16 weights and M >= 6 ----------
TC_FORMATS = FORMATS


@pytest.mark.parametrize("fmt", TC_FORMATS)
@pytest.mark.parametrize("M", [6, 37, 300])
def test_tensor_core_product(orc, fmt, M):
    # N not a multiple of the 128-row tile; M across the 16..256 activation
    # tiles with partial tiles; K = 1280 spans several staged blocks
    N, K = 200, 1280
    w = synth.payload(fmt, (N, K), seed=M)
    x_t, x_bits = _x_bf16(M, K, 7 * M)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "bfloat16")
    _check(_run(fmt, N, K, M, w, x_t, weights="bfloat16"), ref, yabs, K, what=f"{fmt} M={M}")


@pytest.mark.parametrize("fmt,K", [("gguf:q8_0", 96), ("gguf:q4_0", 32), ("q8_g32_fp16", 8192 + 32),
                                   ("gguf:q4_k", 256), ("gguf:q6_k", 14336), ("fp8_e4m3fn_row_fp16", 48)])
def test_tensor_core_ragged_k(orc, fmt, K):
    # K not a multiple of the 64-weight k-step (zero-filled tail), and long K
    N, M = 130, 20
    w = synth.payload(fmt, (N, K), seed=K)
    x_t, x_bits = _x_bf16(M, K, K)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "bfloat16")
    _check(_run(fmt, N, K, M, w, x_t, weights="bfloat16"), ref, yabs, K, what=f"{fmt} K={K}")
    _check(_run(fmt, N, K, M, w, x_t, weights="bfloat16", out_dtype=torch.bfloat16), ref, yabs, K, bf16_out=True,
           what=f"{fmt} K={K} bf16 out")


def test_tensor_core_unaligned_payload_and_determinism(orc):
    fmt, N, K, M = "gguf:q6_k", 256, 2048, 64
    w = synth.payload(fmt, (N, K), seed=3)
    x_t, x_bits = _x_bf16(M, K, 3)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "bfloat16")
    a = _run(fmt, N, K, M, w, x_t, weights="bfloat16", w_off=5)
    _check(a, ref, yabs, K, what="q6_k w+5")
    b = _run(fmt, N, K, M, w, x_t, weights="bfloat16", w_off=5)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt,N,K", [("gguf:q4_k", 1000, 4096), ("gguf:q6_k", 300, 14336), ("gguf:iq4_nl", 1000, 2048)])
def test_tensor_core_split_k_16_rows(orc, fmt, N, K):
    # 16 activation rows per tile: K splits over clusters of up to 8 CTAs
    M = 16
    w = synth.payload(fmt, (N, K), seed=N)
    x_t, x_bits = _x_bf16(M, K, K)
    ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "bfloat16")
    a = _run(fmt, N, K, M, w, x_t, weights="bfloat16")
    _check(a, ref, yabs, K, what=f"{fmt} [{N},{K}] M=16")
    assert np.array_equal(a, _run(fmt, N, K, M, w, x_t, weights="bfloat16"))


def _batched(items, K, M, weights="float32", out=torch.float32, seed=51):
    # items: (fmt, N); returns outputs of the batched call and of single calls
    x_t, x_bits = _x_bf16(M, K, seed)
    x = x_t.to(DEV)
    ws = [(fmt, N, synth.payload(fmt, (N, K), seed=seed + 7 * i)) for i, (fmt, N) in enumerate(items)]
    wd = [torch.from_numpy(w).to(DEV) for _, _, w in ws]
    wdt = torch.float32 if weights == "float32" else torch.bfloat16
    got = ndq.matmul_packed_batched([(fmt, w, N) for (fmt, N, _), w in zip(ws, wd)], K, x, out_dtype=out,
                                    weight_dtype=wdt)
    single = [ndq.matmul_packed(fmt, w, N, K, x, out_dtype=out, weight_dtype=wdt) for (fmt, N, _), w in zip(ws, wd)]
    torch.cuda.synchronize()
    return ws, x_bits, got, single


@pytest.mark.parametrize("items,K", [
    ([("gguf:q4_k", 512), ("gguf:q4_k", 128), ("gguf:q4_k", 128)], 4096),        # q, k, v of a layer
    ([("gguf:q6_k", 1000), ("gguf:q6_k", 1000)], 4096),                          # gate and up
    ([("gguf:q8_0", n) for n in (1, 7, 130, 3, 64, 9, 300, 2)], 4096),           # 8 tensors
    ([("q8_g32_fp16", 33), ("gguf:q8_0", 17)], 2048),                            # one family, two identifiers
    ([("gguf:q8_0", n) for n in (1, 7, 130)], 14336),                            # K > 4096: one call each
])
@pytest.mark.parametrize("weights,out", [("float32", torch.float32), ("bfloat16", torch.bfloat16)])
def test_batched_products_one_launch(orc, items, K, weights, out):
    # one k_gemvl launch over all the products: each output equals the
    # single call's bit for bit (the same per-row summation) and the oracle
    ws, x_bits, got, single = _batched(items, K, 1, weights, out)
    for (fmt, N, w), g, s1 in zip(ws, got, single):
        assert torch.equal(g.view(torch.int32 if out == torch.float32 else torch.int16),
                           s1.view(torch.int32 if out == torch.float32 else torch.int16)), f"{fmt} [{N},{K}]"
        ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, weights)
        _check(g.float().cpu().numpy().astype(np.float64), ref, yabs, K, bf16_out=out == torch.bfloat16,
               what=f"batched {fmt} [{N},{K}]")


@pytest.mark.parametrize("items,K,M", [
    ([("gguf:q4_k", 300), ("gguf:q6_k", 200), ("gguf:iq4_nl", 50)], 4096, 1),     # formats differ
    ([("gguf:q6_k", 300), ("gguf:q8_0", 77)], 4096, 3),                          # three rows of X
    ([("gguf:q4_k", 100)] * 9, 4096, 1),                                          # more than 8 products
    ([("gguf:q4_k", 100), ("gguf:q4_k", 0)], 4096, 1),                            # an empty product
])
def test_batched_products_one_after_another(orc, items, K, M):
    ws, x_bits, got, single = _batched(items, K, M)
    for (fmt, N, w), g, s1 in zip(ws, got, single):
        assert torch.equal(g.view(torch.int32), s1.view(torch.int32)), f"{fmt} [{N},{K}]"
        if N == 0:
            continue
        ref, yabs = orc.matmul_packed(fmt, N, K, w, x_bits, "float32")
        _check(g.cpu().numpy().astype(np.float64), ref, yabs, K, what=f"batched {fmt} [{N},{K}] M={M}")
