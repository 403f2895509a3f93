/*
 * ndq.h -- C ABI of the GB300 (sm_103a) packed quantized-weight decoder.
 *
 * The library decodes packed quantized weight payloads into float tensors
 * under the contract of the ONNX "DequantizePacked decoding specification"
 * (opset 29), section "Signature and storage":
 *
 *     y = DequantizePacked<format, shape, output_dtype>(x)
 *
 * x is the exact payload bytes; blocks are decoded in input order to binary32
 * with the specification's rounding points ("Decoding algorithms": every
 * multiplication, addition and subtraction rounded separately, no fusion),
 * the values are laid out in `shape` (row-major) and converted once to the
 * output type (FLOAT16 / BFLOAT16 by round-to-nearest-even; DOUBLE exactly).
 *
 * Everything runs on the caller's CUDA device and stream.  The header pulls in
 * no CUDA or framework header: streams are passed as `void*` (a cudaStream_t;
 * NULL means the legacy default stream) and buffers as plain pointers.
 *
 * Thread safety: all entry points may be called from several host threads.
 * Calls are asynchronous with respect to the host unless stated otherwise.
 */
#ifndef NDQ_H
#define NDQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Status codes.  Every entry point returns one of these (0 = success).      */
/* Validation errors are returned synchronously before anything is launched. */
/* ------------------------------------------------------------------------ */
#define NDQ_OK 0
#define NDQ_ERR_NULL 1               /* a required pointer is NULL */
#define NDQ_ERR_UNKNOWN_FORMAT 2     /* not one of the registered identifiers */
#define NDQ_ERR_UNSUPPORTED_FORMAT 3 /* registered, but this build has no decoder */
#define NDQ_ERR_BAD_RANK 4           /* ndim < 1 or ndim > NDQ_MAX_RANK */
#define NDQ_ERR_NEGATIVE_DIM 5       /* a dimension is negative */
#define NDQ_ERR_NOT_BLOCK_ALIGNED 6  /* shape[-1] % B != 0 */
#define NDQ_ERR_LENGTH_MISMATCH 7    /* x_len violates the length rule */
#define NDQ_ERR_OVERFLOW 8           /* an element or byte count overflows */
#define NDQ_ERR_BAD_DTYPE 9          /* out_dtype is not one of NDQ_FLOAT.. */
#define NDQ_ERR_WORKSPACE 10         /* batched workspace NULL or too small */
#define NDQ_ERR_CUDA 11              /* a CUDA runtime call or launch failed */
#define NDQ_ERR_DEVICE_FAULT 12      /* a kernel gave up on a bounded wait */
#define NDQ_ERR_BAD_COUNT 13         /* batched tensor count < 0 */
#define NDQ_ERR_TOO_MANY_TENSORS 14  /* no-allocation batch larger than its table */

/* Output element types: the ONNX TensorProto data-type numbers of the four
 * output types DequantizePacked supports ("Signature and storage"). */
#define NDQ_FLOAT 1
#define NDQ_FLOAT16 10
#define NDQ_DOUBLE 11
#define NDQ_BFLOAT16 16

/* Format identifiers: a closed enumeration.  0..26 are the 27 fixed GGUF
 * profiles of "Quantization formats", in the specification's table order;
 * 27..35 are formats of the NInfer "tensor-formats" registry. */
#define NDQ_GGUF_Q4_0 0
#define NDQ_GGUF_Q4_1 1
#define NDQ_GGUF_Q5_0 2
#define NDQ_GGUF_Q5_1 3
#define NDQ_GGUF_Q8_0 4
#define NDQ_GGUF_Q8_1 5
#define NDQ_GGUF_Q2_K 6
#define NDQ_GGUF_Q3_K 7
#define NDQ_GGUF_Q4_K 8
#define NDQ_GGUF_Q5_K 9
#define NDQ_GGUF_Q6_K 10
#define NDQ_GGUF_Q8_K 11
#define NDQ_GGUF_IQ2_XXS 12
#define NDQ_GGUF_IQ2_XS 13
#define NDQ_GGUF_IQ3_XXS 14
#define NDQ_GGUF_IQ1_S 15
#define NDQ_GGUF_IQ4_NL 16
#define NDQ_GGUF_IQ3_S 17
#define NDQ_GGUF_IQ2_S 18
#define NDQ_GGUF_IQ4_XS 19
#define NDQ_GGUF_IQ1_M 20
#define NDQ_GGUF_TQ1_0 21
#define NDQ_GGUF_TQ2_0 22
#define NDQ_GGUF_MXFP4 23
#define NDQ_GGUF_NVFP4 24
#define NDQ_GGUF_Q1_0 25
#define NDQ_GGUF_Q2_0 26
/* nvfp4 (NInfer section 3.3): E2M1 codes, one E4M3FN scale per 16 values and
 * FP32 weight divisors.  Byte layout (a reading: the NInfer page gives the
 * semantics, not the bytes): 64-value blocks of 36 bytes laid out as
 * gguf:nvfp4 (4 scale bytes, then 32 code bytes; group g's codes in bytes
 * 4+8g..11+8g, low nibbles then high nibbles), followed after the last block
 * by D >= 1 little-endian FP32 divisors d_w; row r of the N = prod(shape[:-1])
 * rows uses divisor floor(r / (N / D)), so D must divide N.  Each element is
 * decode_e2m1(c) * decode_e4m3fn(s) rounded once after division by d_w. */
#define NDQ_NVFP4 27
/* q4_g64_fp16 (NInfer sections 4-6.2): 64-value blocks of 34 bytes: a
 * binary16 scale, then 32 bytes holding element k in bits 4*(k mod 2) of byte
 * floor(k/2) as a 4-bit two's-complement code (a layout reading). */
#define NDQ_Q4_G64_FP16 28
/* q8_g32_fp16 (NInfer sections 4-6.2): 32-value blocks of 34 bytes: a
 * binary16 scale then 32 signed bytes (byte-identical to gguf:q8_0). */
#define NDQ_Q8_G32_FP16 29
/* The other grouped signed-integer schemes of NInfer sections 4-6.2.  Each
 * block is one group: a binary16 scale, then the group's G codes of b bits as
 * an LSB-first bit stream (code k in bits [b*k, b*k + b) of the bytes after
 * the scale; a layout reading extending q4_g64_fp16's), so S = 2 + G*b/8.
 * w = binary32(scale * code).
 *   q2_g64_fp16: b = 2, G = 64, code = u - 1 (the Q2_0 grid; byte-identical
 *                to gguf:q2_0);
 *   q5_g64_fp16, q6_g64_fp16: b = 5 / 6, G = 64, two's complement;
 *   t2_g128_fp16: b = 2, G = 128, two's complement (the word 0b10 = -2 is
 *                outside the format and decodes as -2). */
#define NDQ_Q2_G64_FP16 30
#define NDQ_Q5_G64_FP16 31
#define NDQ_Q6_G64_FP16 32
#define NDQ_T2_G128_FP16 33
/* Row-scaled FP8 (NInfer fp8_e4m3fn_row_bf16 / fp8_e4m3fn_row_fp16): one
 * E4M3FN code per element and one multiplier per row, w = binary32(c * s).
 * Layout (a reading): the N*K code bytes of the N = prod(shape[:-1]) rows
 * (row-major), then N little-endian 16-bit multipliers (BF16 or binary16).
 * B = S = 1 (a "block" is one code); x_len = N*K + 2*N, 0 when empty. */
#define NDQ_FP8_E4M3FN_ROW_BF16 34
#define NDQ_FP8_E4M3FN_ROW_FP16 35
#define NDQ_NUM_FORMATS 36

#define NDQ_MAX_RANK 8

/* Map an identifier to its format id ("Format identifiers": case-sensitive,
 * exact; parameterised spellings are unknown).  Returns -1 when unknown or
 * when `id` is NULL. */
int ndq_format_from_name(const char *id);

/* Canonical identifier of a format id ("gguf:q4_k", "nvfp4", ...), or NULL.
 * The string is static and owned by the library. */
const char *ndq_format_name(int format_id);

/* Block geometry of a format: B decoded elements and S packed bytes per block
 * ("Quantization formats" table; NInfer formats as described above).
 * Returns NDQ_ERR_UNKNOWN_FORMAT for an unregistered id, NDQ_ERR_NULL for NULL
 * outputs.  Works for every registered id, decodable or not. */
int ndq_format_geometry(int format_id, int *B, int *S);

/* 1 if this build decodes the format on the GPU, 0 if it is registered but
 * unsupported, -1 if the id is unknown. */
int ndq_format_supported(int format_id);

/* Static, human-readable name of a status code. */
const char *ndq_status_string(int status);

/* Host-only validation of one payload under the length rule of "Signature
 * and storage": rank >= 1, nonnegative dims, shape[-1] % B == 0 and
 * x_len == prod(shape[:-1]) * (shape[-1] / B) * S (for nvfp4 plus 4*D bytes of
 * divisors, D >= 1 dividing the row count; for the fp8 row formats plus 2
 * bytes per row; no trailing words when the tensor is empty).
 * On success writes the block count, the element count and the number of
 * trailing per-row words (nvfp4 divisors, fp8 row multipliers; 0 otherwise);
 * any output pointer may be NULL.  Does not touch the GPU. */
int ndq_payload_geometry(int format_id, const int64_t *shape, int ndim, uint64_t x_len,
                         uint64_t *nblocks, uint64_t *nelements, uint64_t *ndivisors);

/* Decode one payload.
 *   format_id  one of NDQ_* format ids (must be supported by this build)
 *   shape      host array of ndim logical dimensions (ONNX order: the last
 *              dimension is contiguous and is the block axis)
 *   out_dtype  NDQ_FLOAT, NDQ_FLOAT16, NDQ_BFLOAT16 or NDQ_DOUBLE
 *   x_u8       device pointer to x_len payload bytes (any alignment; a
 *              16-byte-aligned payload takes the bulk-copy path)
 *   y          device pointer receiving prod(shape) elements of out_dtype,
 *              row-major (any alignment; 16-byte alignment takes the vector
 *              store path)
 *   stream     cudaStream_t to enqueue on (NULL = legacy default stream)
 * The caller owns x and y and keeps them alive until the stream has passed
 * the call.  The call allocates nothing and is asynchronous; validation
 * errors return before any launch; an empty tensor returns NDQ_OK without a
 * launch; a launch failure returns NDQ_ERR_CUDA.  No payload byte is
 * rejected: every bit pattern decodes to a defined value (NaN/inf scales
 * propagate by IEEE rules).  x and y must not overlap. */
int ndq_dequantize_packed(int format_id, const int64_t *shape, int ndim, int out_dtype,
                          const uint8_t *x_u8, size_t x_len, void *y, void *stream);

/* One tensor of a batched decode (same meaning as the single call's
 * arguments; x and y are device pointers). */
typedef struct ndq_tensor_desc {
    int32_t format_id;
    int32_t ndim;
    int64_t shape[NDQ_MAX_RANK];
    int32_t out_dtype;
    int32_t reserved; /* ignored; set to 0 */
    const uint8_t *x;
    uint64_t x_len;
    void *y;
} ndq_tensor_desc;

/* Decode fused into a matrix product (the consumer-side use of a packed
 * weight: NInfer "tensor-formats" lets a consuming kernel fuse decode into
 * its product with its own staging, reduction order and precision):
 *
 *     Y[m, n] = sum_k X[m, k] * W[n, k]      (m < M, n < N, k < K)
 *
 *   format_id     any supported format (the fp8 row formats need K % 16 == 0)
 *   w, w_len      device payload of the weight matrix [N, K] under the same
 *                 length rule as ndq_dequantize_packed
 *   x_bf16        device bfloat16 activations [M, K], row-major
 *   weight_dtype  NDQ_FLOAT: W is the payload decoded exactly as
 *                 ndq_dequantize_packed decodes it to FLOAT; NDQ_BFLOAT16: W
 *                 is that decode rounded once to bfloat16 (the operand of an
 *                 unfused decode-to-bf16 and bf16 product)
 *   y             device output [M, N], row-major, NDQ_FLOAT or NDQ_BFLOAT16
 * Products and sums are binary32 in an unspecified but fixed order, so
 * repeated calls give identical bits; each output is within
 * 2*(K+16)*2^-24 * sum_k |X[m,k] W[n,k]| of the exact sum, then rounded once
 * to out_dtype.  Kernels: one row of X on the CUDA cores (fused
 * multiply-adds); with NDQ_BFLOAT16 weights, 6 or more rows, X 16-byte
 * aligned and K % 8 == 0, on the tensor cores (tcgen05, binary32
 * accumulation in tensor memory) in one pass; otherwise up to 8 rows of
 * gguf q8_0, q8_g32_fp16, q4_k or q6_k with K % 512 == 0 and 16-byte-aligned
 * payload rows on the CUDA cores with X held in shared memory when it fits
 * (each weight decoded once for all the rows; for one row only when
 * K > 4096, shorter rows keeping X in registers); 2 to 8 rows with
 * NDQ_FLOAT weights of gguf q6_k, q8_0 or q8_g32_fp16, X 16-byte aligned
 * and K % 8 == 0, on the tensor cores with the group scales applied to the
 * tensor core's per-group sums; other cases up to 8 rows per pass on the
 * CUDA cores (each pass reads the payload once).  Same ownership, asynchrony and error
 * rules as ndq_dequantize_packed; M, N or K of 0 is valid (K == 0 writes
 * zeros); NDQ_ERR_BAD_DTYPE for other weight or output types. */
int ndq_matmul_packed(int format_id, int64_t N, int64_t K, const uint8_t *w, size_t w_len, const void *x_bf16,
                      int64_t M, int weight_dtype, int out_dtype, void *y, void *stream);

/* One product of a batched fused call: weight payload w [n, K] (device,
 * w_len bytes, same length rule as ndq_matmul_packed) and its output y
 * [M, n] (device). */
typedef struct ndq_matmul_desc {
    int32_t format_id;
    int32_t reserved; /* ignored; set to 0 */
    int64_t n;
    const uint8_t *w;
    uint64_t w_len;
    void *y;
} ndq_matmul_desc;

/* Several fused products that share their activations X [M, K]:
 * y_i = X * W_i^T for every descriptor, exactly as `count` calls of
 * ndq_matmul_packed with the same x_bf16, K, M, weight_dtype and out_dtype
 * (the same bounds; each output is the same as that call's in every bit
 * when it takes the same kernel).  This is not part of the DequantizePacked
 * specification: it lets the weights that read one activation row (a
 * layer's q, k and v projections, or its gate and up projections) run as
 * ONE kernel launch when M == 1, count <= 8, every product has n > 0 and
 * the same format, K % 512 == 0, K <= 4096, the format is gguf q8_0 /
 * q8_g32_fp16 / q4_k / q6_k and every payload row starts on a 16-byte
 * boundary; otherwise the products are launched one after another.
 *   descs  host array of `count` descriptors, read during the call only
 * Every descriptor is validated before anything is launched (the status of
 * the first invalid one is returned: the codes of ndq_matmul_packed, or
 * NDQ_ERR_BAD_COUNT for count < 0); count == 0 returns NDQ_OK.  Allocates
 * nothing; asynchronous on `stream` like ndq_matmul_packed. */
int ndq_matmul_packed_batched(const ndq_matmul_desc *descs, int count, int64_t K, const void *x_bf16, int64_t M,
                              int weight_dtype, int out_dtype, void *stream);

/* Device workspace bytes the batched call needs for n tensors (a table of
 * per-tensor launch descriptors), or 0 when n < 0. */
size_t ndq_batched_workspace_bytes(int n);

/* Decode n tensors (for example every weight of a model) in ONE kernel
 * launch.  This is not part of the DequantizePacked specification: it is a
 * launcher over the same per-tensor decode.
 *   descs      host array of n descriptors; read during the call only
 *   workspace  device buffer of at least ndq_batched_workspace_bytes(n) bytes,
 *              16-byte aligned; the call writes the launch table into it with
 *              one cudaMemcpyAsync on `stream` and the kernel reads it, so the
 *              caller keeps it alive and unmodified until the stream has
 *              passed the call, and does not share it between calls that may
 *              run concurrently
 *   stream     as for the single call
 * Every descriptor is validated before anything is enqueued: one bad entry
 * rejects the whole batch with that entry's status.  Outputs of different
 * tensors must not overlap each other or any payload.  n == 0, or a batch
 * whose tensors are all empty, returns NDQ_OK without a launch. */
int ndq_dequantize_packed_batched(const ndq_tensor_desc *descs, int n, void *workspace,
                                  size_t ws_bytes, void *stream);

/* Largest batch the no-allocation variant below accepts. */
#define NDQ_NOALLOC_MAX_TENSORS 1024

/* Batched decode for callers that cannot allocate device memory.  (There is
 * no counterpart on the pages: this is a convenience of this library.)
 *
 * Some callers cannot call cudaMalloc or any other allocator: a plain C or
 * plugin host embedded in a process whose device memory is reserved up front
 * by another framework's pool, or a runtime with a fixed memory budget, where
 * an extra allocation would fail, fragment the pool or synchronize the
 * device.  For them this entry point does the same work as
 * ndq_dequantize_packed_batched without a workspace argument: the launch
 * table is kept in a fixed device array inside the library (room for
 * NDQ_NOALLOC_MAX_TENSORS non-empty tensors, 64 bytes each, i.e. 64 KiB that
 * every GPU which loads the library holds until the process exits).  The
 * caller still passes every input and output (descs[i].x and descs[i].y).
 *   descs   host array of n descriptors (same meaning as for the batched
 *           call), read during the call only
 *   stream  cudaStream_t to enqueue on (NULL = legacy default stream)
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  The first call on a device looks up the array's device address
 * with cudaGetSymbolAddress while that device is current; make that first
 * call before any stream capture.  Every call rewrites the part of the table
 * it uses, and the array keeps the last call's contents; calls whose work may
 * overlap on the GPU (different streams or host threads without ordering)
 * share the array and race, so order them on one stream.
 * Errors: n > NDQ_NOALLOC_MAX_TENSORS returns NDQ_ERR_TOO_MANY_TENSORS before
 * anything is enqueued; n < 0 returns NDQ_ERR_BAD_COUNT; otherwise the same
 * validation and errors as ndq_dequantize_packed_batched (minus workspace). */
int ndq_dequantize_packed_batched_noalloc(const ndq_tensor_desc *descs, int n, void *stream);

/* Failure-path check (not part of the pages' contract): makes the NEXT decode
 * launch issued by the calling host thread (ndq_dequantize_packed or a
 * batched call) exercise its device-side failure path without any GPU fault.
 * That launch withholds the staging copy of global tile `tile` (the tiles of
 * a launch are its tensors' 8192-element spans in order), so the decode
 * warps waiting for that tile give up after `wait_limit_us` microseconds
 * instead of the default 2 s, set their bits in the device fault word and
 * stop; the CTA's producer then gives up too, waits for every copy it did
 * issue, and stops.  Every other CTA decodes its tiles normally.  The
 * request is consumed by that one launch (a launch of no tile does not
 * consume it); tile = -1 cancels it.  Outputs of the affected CTA's tiles are
 * unspecified; read the fault word with ndq_get_device_fault afterwards.
 * Returns NDQ_ERR_BAD_COUNT when tile < -1 or wait_limit_us is 0 or above
 * 2000000. */
int ndq_test_withhold_copy(int64_t tile, uint32_t wait_limit_us);

/* Read and clear the library's device fault word on the current device.
 * A kernel sets a nonzero bit when one of its bounded waits for staged
 * payload data gives up (it then stops decoding instead of hanging the GPU).
 * This call synchronizes the device.  *flags == 0 means no fault occurred
 * since the last call.  Returns NDQ_ERR_CUDA if the device cannot be read. */
int ndq_get_device_fault(uint32_t *flags);

#ifdef __cplusplus
}
#endif

#endif /* NDQ_H */
