// ndq_internal.h -- launch descriptors shared by the host ABI (ndq_api.cpp)
// and the decode kernels (ndq_kernels.cu).  Not part of the public ABI.
// The fused product's descriptors are in ndq_fused.h.
#pragma once

#include <cstddef>
#include <cstdint>

namespace ndq {

// Kernel decode families.  gguf:q8_0 and q8_g32_fp16 share one (their blocks
// are byte- and value-identical).
enum KFmt : int32_t {
    KF_Q8_0 = 0,
    KF_Q4_0 = 1,
    KF_IQ4_NL = 2,
    KF_Q4_K = 3,
    KF_Q6_K = 4,
    KF_MXFP4 = 5,
    KF_GGUF_NVFP4 = 6,
    KF_NVFP4 = 7,
    KF_Q4_G64 = 8,
    KF_Q4_1 = 9,
    KF_Q5_0 = 10,
    KF_Q5_1 = 11,
    KF_Q8_1 = 12,
    KF_Q8_K = 13,
    KF_Q2_K = 14,
    KF_Q3_K = 15,
    KF_Q5_K = 16,
    KF_IQ4_XS = 17,
    KF_TQ1_0 = 18,
    KF_TQ2_0 = 19,
    KF_Q1_0 = 20,
    KF_Q2_0 = 21,
    KF_IQ2_XXS = 22,
    KF_IQ2_XS = 23,
    KF_IQ2_S = 24,
    KF_IQ3_XXS = 25,
    KF_IQ3_S = 26,
    KF_IQ1_S = 27,
    KF_IQ1_M = 28,
    KF_Q5_G64 = 29,
    KF_Q6_G64 = 30,
    KF_T2_G128 = 31,
    KF_FP8_ROW_BF16 = 32,
    KF_FP8_ROW_FP16 = 33,
    KF_COUNT = 34,
};

// Format selector of a launch whose tensors mix only gguf:q8_0, gguf:q4_k and
// gguf:q6_k (the usual K-quant model mix): a kernel with just those decoders.
constexpr int32_t kFselKQuantMix = -2;

// Output element type of a tensor.
enum KOut : int32_t { KO_F32 = 0, KO_F16 = 1, KO_BF16 = 2, KO_F64 = 3 };

// Work unit: a tile of kTileElems consecutive output elements (a whole number
// of blocks for every format, since every B divides 8192).  A tile's payload
// span is (8192 / B) * S bytes: a multiple of 16 for every supported format,
// so full tiles of a 16-byte-aligned payload are bulk-copyable.
constexpr int kTileElems = 8192;
constexpr int kThreads = 256;
constexpr int kMaxTileBytes = 9344;  // gguf:q8_k: 32 blocks * 292 bytes
constexpr int kBlockThreads = kThreads + 32;  // consumer warps + one producer warp
constexpr int kConsumerWarpsPerCta = kThreads / 32;
constexpr int kStages = 4;                    // staged tiles in flight per CTA
constexpr int kInStride = 9472;               // tile bytes + phase + rounding + over-read
constexpr int kTabEntries = 256 * 16;         // nvfp4 quotient table (floats)

// Launches whose tensors are all nvfp4 with one 16-bit output type decode by
// byte-table lookup: the 16-bit output of every (scale byte, code) pair,
// built per CTA in the shared-memory region of the nvfp4 quotient table (4 KB
// of its 16 KB).  (gguf:nvfp4 and gguf:mxfp4 have the same structure without
// the division and measured as fast with their 16-entry value table.)
#if defined(__CUDACC__)
#define NDQ_HOST_DEVICE __host__ __device__
#else
#define NDQ_HOST_DEVICE
#endif
NDQ_HOST_DEVICE constexpr bool uses_lut16(int fsel, int osel) {
    return fsel == KF_NVFP4 && (osel == KO_F16 || osel == KO_BF16);
}
// Decode kernels whose output type is 16-bit (or mixed) stage each warp's
// share of a full tile in shared memory and write it with one bulk copy
// (measured faster for most formats), except those measured faster storing
// from registers: the k-quant mix kernel, gguf:q4_k, gguf:q4_0 and nvfp4.
NDQ_HOST_DEVICE constexpr bool decode_staged(int fsel, int osel) {
    return fsel != kFselKQuantMix && fsel != KF_Q4_K && fsel != KF_Q4_0 && fsel != KF_NVFP4 &&
           (osel < 0 || osel == KO_F16 || osel == KO_BF16);
}
// Payload stages in flight per decode CTA: 4 for the kernels that run two
// CTAs per SM (the launches that mix formats, and the q6_k and fp8 row
// decoders, whose 16-bit variants need more than 75 registers) and for
// gguf:q4_0 (no output staging, so 4 stages still fit three CTAs per SM:
// [4096,4096] -> bf16 measured 9.3 us with 3 and 8.6 us with 4), else 3
// (q4_g64, q4_k and the others measured 2-7 % slower with 4).
NDQ_HOST_DEVICE constexpr int decode_stages(int fsel) {
    return (fsel < 0 || fsel == KF_Q6_K || fsel == KF_FP8_ROW_BF16 || fsel == KF_FP8_ROW_FP16 || fsel == KF_Q4_0) ? 4
                                                                                                                    : 3;
}
// Resident CTAs per SM for launches that mix formats (the whole-model decode):
// measured fastest at 2 even when registers and shared memory allow 3.
// Single-format launches use every CTA the occupancy calculator allows.
constexpr int kMixedCtasPerSm = 2;

// One tensor as the kernel sees it (64 bytes; kept trivially copyable).
struct DevTensor {
    const uint8_t* x;         // payload blocks
    void* y;                  // output
    uint64_t nblocks;         // blocks in the payload
    uint64_t tile_begin;      // first global tile index of this tensor
    const uint8_t* divs;      // nvfp4: FP32 divisor words; fp8 rows: the row multipliers (may be unaligned)
    uint64_t blocks_per_div;  // nvfp4: blocks sharing one divisor; fp8 rows: elements per row
    int32_t fmt;              // KFmt
    int32_t out;              // KOut
    uint16_t S;               // bytes per block
    uint16_t B;               // elements per block
    uint16_t bpt;             // blocks per tile (kTileElems / B)
    uint16_t yvec;            // 1 if y is 16-byte aligned
};
static_assert(sizeof(DevTensor) == 64, "DevTensor layout");

// Codebook rows of the IQ2 / IQ3 / IQ1 formats in the layout the kernels
// read: row r of an 8-wide table in one 64-bit word, of a 4-wide table in one
// 32-bit word, entry j in byte j.  iq1s_grid's entries v in {-1, 0, 1} are
// stored as 8 * (v + 1).  One copy per device (see launch_decode).
struct IqGrids {
    uint64_t iq2xxs[256];  // 8, 25 or 43
    uint64_t iq2xs[512];
    uint64_t iq2s[1024];
    uint32_t iq3xxs[256];  // 4, 12, ..., 52, 62
    uint32_t iq3s[512];    // 1, 3, ..., 15
    uint64_t iq1s[2048];   // 0, 8 or 16
};

// Kernel parameters.  A single-tensor launch carries its descriptor inline
// (table == nullptr, n == 1); a batched launch points at a device table of n
// descriptors sorted by tile_begin.
struct KParams {
    DevTensor single;
    const DevTensor* table;
    int32_t n;
    int32_t nv_index;  // first nvfp4 tensor of the launch (its divisor seeds the quotient table), or -1
    uint64_t total_tiles;
    int32_t fsel;      // KFmt shared by every tensor of the launch, kFselKQuantMix, or -1
    int32_t osel;      // KOut shared by every tensor of the launch, or -1
    unsigned int* fault;  // device fault word (set by the launcher)
    const IqGrids* grids;  // IQ codebooks (set by the launcher)
    uint64_t wait_ns;      // limit of the kernel's bounded waits (set by the launcher)
    int64_t withhold_tile;  // tile whose copy the producer withholds, or -1 (set by the launcher)
};

using KernelFn = void (*)(KParams);

// Device addresses of the fault word and the IQ codebooks on the current
// device (resolved once per device).  Returns 0 or a CUDA error code.
int device_symbols(int dev, unsigned int** fault, const IqGrids** grids);

// Kernel getters, one per instantiation file (osel: KOut, or -1 for any).
KernelFn kernel_q8_0(int osel);
KernelFn kernel_q4_0(int osel);
KernelFn kernel_iq4_nl(int osel);
KernelFn kernel_q4_k(int osel);
KernelFn kernel_q6_k(int osel);
KernelFn kernel_mxfp4(int osel);
KernelFn kernel_gguf_nvfp4(int osel);
KernelFn kernel_nvfp4(int osel);
KernelFn kernel_q4_g64(int osel);
KernelFn kernel_q4_1(int osel);
KernelFn kernel_q5_0(int osel);
KernelFn kernel_q5_1(int osel);
KernelFn kernel_q8_1(int osel);
KernelFn kernel_q8_k(int osel);
KernelFn kernel_q2_k(int osel);
KernelFn kernel_q3_k(int osel);
KernelFn kernel_q5_k(int osel);
KernelFn kernel_iq4_xs(int osel);
KernelFn kernel_tq1_0(int osel);
KernelFn kernel_tq2_0(int osel);
KernelFn kernel_q1_0(int osel);
KernelFn kernel_q2_0(int osel);
KernelFn kernel_iq2_xxs(int osel);
KernelFn kernel_iq2_xs(int osel);
KernelFn kernel_iq2_s(int osel);
KernelFn kernel_iq3_xxs(int osel);
KernelFn kernel_iq3_s(int osel);
KernelFn kernel_iq1_s(int osel);
KernelFn kernel_iq1_m(int osel);
KernelFn kernel_q5_g64(int osel);
KernelFn kernel_q6_g64(int osel);
KernelFn kernel_t2_g128(int osel);
KernelFn kernel_fp8_row_bf16(int osel);
KernelFn kernel_fp8_row_fp16(int osel);
KernelFn kernel_generic_f32();
KernelFn kernel_generic_f16();
KernelFn kernel_generic_bf16();
KernelFn kernel_generic_f64();
KernelFn kernel_generic_any();
KernelFn kernel_generic(int osel);
KernelFn kernel_kquant_mix(int osel);

// Dynamic shared memory of a decode CTA: with or without the nvfp4 tables
// (lut: the 4 KB byte table instead of the 16 KB quotient table), and with
// or without the 16-bit output buffers.
size_t decode_smem_bytes(bool tab, bool lut, bool staged, int stages);

// Launch one decode over p.total_tiles tiles on `stream` (a cudaStream_t).
// Returns 0 or a CUDA error code.
int launch_decode(const KParams& p, void* stream);

// Failure-path check of the calling host thread's next decode launch: the
// producer withholds the copy of `tile` and every bounded wait gives up
// after `wait_ns`.  Consumed (reset) by that launch.
void set_withhold_next(int64_t tile, uint64_t wait_ns);

// Launch-table upload: descriptors travel to the device as the parameters of
// a small kernel, kUploadChunk per launch (no host-blocking copy).
constexpr int kUploadChunk = 128;
struct UploadParams {
    DevTensor* dst;  // device entries dst[0..n) are written
    int32_t n;
    DevTensor d[kUploadChunk];
};

// One upload launch on `stream`.  Returns 0 or a CUDA error code.
int upload_chunk(const UploadParams& up, void* stream);

// Copy n host descriptors into a device table with upload launches on
// `stream`.  Returns 0 or a CUDA error code.
int upload_table(DevTensor* dst, const DevTensor* src, int n, void* stream);

// Capacity of the library-owned launch table of the no-allocation batched
// call (64 bytes per entry: 64 KiB per device).
constexpr int kNoAllocMaxTensors = 1024;

// Device address of the library-owned launch table on the current device,
// looked up with cudaGetSymbolAddress on the first call per device.  Returns
// 0 or a CUDA error code.
int noalloc_table(DevTensor** table);

// Kernel selectors of a launch, accumulated over its tensors: the shared
// format (or kFselKQuantMix, or -1) and the shared output type (or -1).
struct KernelSelect {
    int32_t fsel = -3;  // -3: no tensor yet
    int32_t osel = -3;
    bool kmix = true;   // every tensor is gguf:q8_0, q4_k or q6_k
    void add(const DevTensor& t) {
        fsel = (fsel == -3 || fsel == t.fmt) ? t.fmt : -1;
        osel = (osel == -3 || osel == t.out) ? t.out : -1;
        kmix = kmix && (t.fmt == KF_Q8_0 || t.fmt == KF_Q4_K || t.fmt == KF_Q6_K);
    }
    void get(int32_t* f, int32_t* o) const {
        *f = (fsel < 0 && kmix) ? kFselKQuantMix : fsel;
        *o = osel;
    }
};

// Kernel selectors of a launch over tensors t[0..n).
void select_kernel(const DevTensor* t, int n, int32_t* fsel, int32_t* osel);

// Read and clear the device fault word of the current device.
int read_fault(uint32_t* flags);

}  // namespace ndq
