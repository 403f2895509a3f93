// ndq_kernels.cu -- launcher of the decode kernels: kernel selection,
// occupancy-sized persistent grids, the launch-table upload, the library-owned
// table of the no-allocation batched call and the device fault word.  The
// decode kernels themselves are in ndq_device.cuh, instantiated by
// ndq_inst_*.cu.

#include <cuda_runtime.h>

#include <cstdint>

#include "ndq_internal.h"
#include "ndq_iq_codebooks.h"

namespace ndq {

// Set by a kernel whose bounded wait gave up (see ndq_get_device_fault).
__device__ unsigned int g_fault_word;

// The IQ codebooks, expanded at compile time.
__device__ const IqGrids g_iq_grids = iqcb::make_iq_grids();

namespace {

// Writes n descriptors (kernel parameters) into a device table.
__global__ void k_upload_table(const UploadParams p) {
    for (int i = threadIdx.x; i < p.n; i += blockDim.x) p.dst[i] = p.d[i];
}

// Specialised kernels live in one instantiation file per format.
KernelFn pick_kernel(int fsel, int osel) {
    if (osel < 0) return kernel_generic(-1);
    if (fsel == kFselKQuantMix) return kernel_kquant_mix(osel);
    switch (fsel) {
        case KF_Q8_0: return kernel_q8_0(osel);
        case KF_Q4_0: return kernel_q4_0(osel);
        case KF_IQ4_NL: return kernel_iq4_nl(osel);
        case KF_Q4_K: return kernel_q4_k(osel);
        case KF_Q6_K: return kernel_q6_k(osel);
        case KF_MXFP4: return kernel_mxfp4(osel);
        case KF_GGUF_NVFP4: return kernel_gguf_nvfp4(osel);
        case KF_NVFP4: return kernel_nvfp4(osel);
        case KF_Q4_G64: return kernel_q4_g64(osel);
        case KF_Q4_1: return kernel_q4_1(osel);
        case KF_Q5_0: return kernel_q5_0(osel);
        case KF_Q5_1: return kernel_q5_1(osel);
        case KF_Q8_1: return kernel_q8_1(osel);
        case KF_Q8_K: return kernel_q8_k(osel);
        case KF_Q2_K: return kernel_q2_k(osel);
        case KF_Q3_K: return kernel_q3_k(osel);
        case KF_Q5_K: return kernel_q5_k(osel);
        case KF_IQ4_XS: return kernel_iq4_xs(osel);
        case KF_TQ1_0: return kernel_tq1_0(osel);
        case KF_TQ2_0: return kernel_tq2_0(osel);
        case KF_Q1_0: return kernel_q1_0(osel);
        case KF_Q2_0: return kernel_q2_0(osel);
        case KF_IQ2_XXS: return kernel_iq2_xxs(osel);
        case KF_IQ2_XS: return kernel_iq2_xs(osel);
        case KF_IQ2_S: return kernel_iq2_s(osel);
        case KF_IQ3_XXS: return kernel_iq3_xxs(osel);
        case KF_IQ3_S: return kernel_iq3_s(osel);
        case KF_IQ1_S: return kernel_iq1_s(osel);
        case KF_IQ1_M: return kernel_iq1_m(osel);
        case KF_Q5_G64: return kernel_q5_g64(osel);
        case KF_Q6_G64: return kernel_q6_g64(osel);
        case KF_T2_G128: return kernel_t2_g128(osel);
        case KF_FP8_ROW_BF16: return kernel_fp8_row_bf16(osel);
        case KF_FP8_ROW_FP16: return kernel_fp8_row_fp16(osel);
        default: return kernel_generic(osel);
    }
}

constexpr int kKernelSlots = (KF_COUNT + 2) * 5;

int slot_of(int fsel, int osel) { return (osel < 0) ? 0 : (fsel + 2) * 5 + osel + 1; }

struct DeviceInfo {
    int sms = 0;
    int ctas_per_sm[kKernelSlots][2] = {};  // 0 = not yet queried
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];


// Device addresses of the fault word and the IQ codebooks, resolved once per
// device.
unsigned int* g_fault_addr[kMaxDevices];
const IqGrids* g_grids_addr[kMaxDevices];

// Limit of the decode kernels' bounded waits (2 s), and the failure-path
// check requested for this host thread's next launch (none: -1).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
thread_local uint64_t t_wait_ns = kDefaultWaitNs;
thread_local int64_t t_withhold_tile = -1;

}  // namespace

void set_withhold_next(int64_t tile, uint64_t wait_ns) {
    t_withhold_tile = tile;
    t_wait_ns = wait_ns;
}

int launch_decode(const KParams& p, void* stream) {
    if (p.total_tiles == 0) return 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
    const int fsel = ((p.fsel >= 0 && p.fsel < KF_COUNT) || p.fsel == kFselKQuantMix) ? p.fsel : -1;
    const int osel = (p.osel >= 0 && p.osel <= KO_F64) ? p.osel : -1;
    const bool lut = uses_lut16(fsel, osel), staged = decode_staged(fsel, osel);
    const int stages = decode_stages(fsel);
    const bool tab = p.nv_index >= 0 || lut;
    const size_t smem = decode_smem_bytes(tab, lut, staged, stages);
    const KernelFn fn = pick_kernel(fsel, osel);
    if (!fn) return static_cast<int>(cudaErrorInvalidDeviceFunction);
    DeviceInfo& di = g_dev[dev];
    // Benign race: concurrent first calls compute and store the same values.
    if (di.sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return static_cast<int>(e);
        di.sms = sms;
    }
    int& cps = di.ctas_per_sm[slot_of(fsel, osel)][tab ? 1 : 0];
    if (cps == 0) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(decode_smem_bytes(true, lut, staged, stages)));
        if (e != cudaSuccess) return static_cast<int>(e);
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kBlockThreads, smem);
        if (e != cudaSuccess) return static_cast<int>(e);
        if (fsel < 0 && n > kMixedCtasPerSm) n = kMixedCtasPerSm;
        cps = n > 0 ? n : 1;
    }
    KParams q = p;
    const int se = device_symbols(dev, &q.fault, &q.grids);
    if (se != 0) return se;
    q.wait_ns = t_wait_ns;
    q.withhold_tile = t_withhold_tile;
    t_wait_ns = kDefaultWaitNs;  // a requested failure-path check applies to one launch
    t_withhold_tile = -1;
    const uint64_t resident = static_cast<uint64_t>(di.sms) * static_cast<uint64_t>(cps);
    const unsigned grid = static_cast<unsigned>(p.total_tiles < resident ? p.total_tiles : resident);
    void* args[] = {&q};
    // programmatic stream serialization: the kernel waits on the previous
    // grid itself (griddepcontrol.wait), so its CTAs may be placed as soon as
    // the previous grid's CTAs retire
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBlockThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(fn), args);
    return static_cast<int>(e);
}

int device_symbols(int dev, unsigned int** fault, const IqGrids** grids) {
    if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
    if (!g_fault_addr[dev]) {
        void* addr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&addr, g_fault_word);
        if (e != cudaSuccess) return static_cast<int>(e);
        g_fault_addr[dev] = static_cast<unsigned int*>(addr);
    }
    if (!g_grids_addr[dev]) {
        void* addr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&addr, g_iq_grids);
        if (e != cudaSuccess) return static_cast<int>(e);
        g_grids_addr[dev] = static_cast<const IqGrids*>(addr);
    }
    *fault = g_fault_addr[dev];
    *grids = g_grids_addr[dev];
    return 0;
}

int upload_chunk(const UploadParams& up, void* stream) {
    k_upload_table<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(up);
    return static_cast<int>(cudaGetLastError());
}

int upload_table(DevTensor* dst, const DevTensor* src, int n, void* stream) {
    for (int i0 = 0; i0 < n; i0 += kUploadChunk) {
        UploadParams up;
        up.dst = dst + i0;
        up.n = (n - i0) < kUploadChunk ? (n - i0) : kUploadChunk;
        for (int i = 0; i < up.n; ++i) up.d[i] = src[i0 + i];
        const int e = upload_chunk(up, stream);
        if (e != 0) return e;
    }
    return 0;
}

// ---------------------------------------------------------------------------
// The launch table of the no-allocation batched call: a fixed file-scope
// device array (kNoAllocMaxTensors entries, 64 KiB) that every GPU which
// loads this library holds until process exit.  The host cannot use the
// array's name as a device address, so its address is looked up once per
// device with cudaGetSymbolAddress while that device is current.  Every call
// overwrites entries [0, n) before its decode launch on the same stream;
// nothing has to start at zero because the decode reads only the n entries
// that call wrote.  Calls whose work overlaps on the GPU (other streams,
// other host threads) share the array and race.
// ---------------------------------------------------------------------------
static __device__ __align__(256) DevTensor g_noalloc_table[kNoAllocMaxTensors];

namespace {
DevTensor* g_noalloc_addr[kMaxDevices];  // per-device address, set once
}

int noalloc_table(DevTensor** table) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= kMaxDevices) return static_cast<int>(cudaErrorInvalidDevice);
    if (!g_noalloc_addr[dev]) {  // first call on this device: resolve the symbol
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_table);
        if (e != cudaSuccess) return static_cast<int>(e);
        g_noalloc_addr[dev] = static_cast<DevTensor*>(addr);
    }
    *table = g_noalloc_addr[dev];
    return 0;
}

void select_kernel(const DevTensor* t, int n, int32_t* fsel, int32_t* osel) {
    KernelSelect sel;
    for (int i = 0; i < n; ++i) sel.add(t[i]);
    sel.get(fsel, osel);
}

int read_fault(uint32_t* flags) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return static_cast<int>(e);
    *flags = v;
    return 0;
}

}  // namespace ndq
