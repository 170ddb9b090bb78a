// gemm_i8_run_noalloc: the int8 GEMM without any device-memory allocation.
//
// Who needs it: callers that are not allowed to allocate device memory
// themselves or through a library they call — runtimes that plan every byte
// of device memory up front and forbid libraries to grab more, and
// latency-critical loops where an allocation could block, synchronise the
// device or fail part-way through a run.  gemm_i8_run takes its f16 operand
// copies from a stream-ordered pool; this entry point uses instead a fixed
// scratch array that lives in the library's own device image.
//
// The scratch is a file-scope static __device__ array of kNoAllocScratchBytes
// (64 MiB).  Every GPU that loads the library holds it until the process
// exits, whether or not this entry point is ever called.  In host code the
// array's name is only a host-side stand-in, not a device address, so the
// first call on each device (with that device current) looks its device
// address up with cudaGetSymbolAddress and caches it; that first call should
// come before any stream capture.
//
// All calls share the one array and it keeps the last call's contents.  The
// staging kernel (or, on the skinny path, the prologue that writes the f16
// copy of A) overwrites every element the GEMM reads (the pad columns of each
// row are never read).  Calls whose work overlaps on the GPU (on different
// streams, or on different host threads without ordering) race on the array
// and give wrong results: order them.
//
// A kernel wait that runs past its limit records its code in the device error
// word that every entry point shares (itself a static __device__ variable, so
// no allocation either); gemm_device_error reads and clears it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/dense_int8_matrix.h"
#include "internal.h"

namespace gemm {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // GEMM_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The skinny path's f16 copy of A (m <= 128 rows, k <= GEMM_I8_MAX_K) always
// fits the array.
static_assert(int64_t(128) * GEMM_I8_MAX_K * 2 <= int64_t(kNoAllocScratchBytes),
              "skinny f16 activations must fit the static scratch");

constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int tc2_pairs = 0;                  // co-resident pairs of the two-SM kernel
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
    int* err = nullptr;                 // device address of the shared error word
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Once per device, with the device current: attributes and the device
// addresses of the static arrays.  No allocation.
gemm_status noalloc_device(NoAllocDevice** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
            d.scratch = static_cast<unsigned char*>(p);
            if (device_error_word(&d.err) != cudaSuccess) return GEMM_ERR_CUDA;
            d.tc2_pairs = tc2_max_pairs();
        }
        d.ready = true;
    }
    *out = &d;
    return GEMM_OK;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace

}  // namespace gemm

extern "C" gemm_status gemm_i8_run_noalloc(const gemm_plan* p, const int8_t* A, const int8_t* Bt, int32_t* C,
                                           void* stream_ptr) {
    using namespace gemm;
    // the same plan and pointer checks as gemm_i8_run, then the scratch limit
    gemm_status st = check_plan(p, GEMM_DTYPE_I8);
    if (st != GEMM_OK) return st;
    st = check_ptrs(A, Bt, C);
    if (st != GEMM_OK) return st;
    const bool skinny = p->path == GEMM_PATH_SKINNY;
    if (skinny) {
        // f16 copy of A on the tensor-core skinny kernel (m * k * 2 bytes)
        if (p->k > GEMM_I8_MAX_K || p->m * p->k * 2 > static_cast<int64_t>(kNoAllocScratchBytes))
            return GEMM_ERR_INVALID_ARG;
    } else {
        // the f16 copies of A and Bt must fit the static scratch array
        const int64_t need = round256(p->m * p->k_pitch * 2) + round256(p->n * p->k_pitch * 2);
        if (need > static_cast<int64_t>(kNoAllocScratchBytes)) return GEMM_ERR_INVALID_ARG;
    }
    NoAllocDevice* d = nullptr;
    st = noalloc_device(&d);
    if (st != GEMM_OK) return st;
    if (!d->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    if (skinny) {
        if (skinny_tc_supported(p->m, p->n, p->k, A, Bt) && tensor_map_encoder_available()) {
            // as in gemm_i8_run, with the f16 copy of A (m * k * 2 <= 32 MiB for
            // any k the planner accepts) at the start of the static array
            uint16_t* A16 = reinterpret_cast<uint16_t*>(d->scratch);
            if (launch_skinny_prologue(A, A16, C, p->m, p->n, p->k, d->num_sms, stream) != cudaSuccess ||
                launch_skinny_tc(Bt, A16, C, d->err, p->m, p->n, p->k, d->num_sms, stream) != cudaSuccess)
                return GEMM_ERR_CUDA;
            return GEMM_OK;
        }
        return launch_skinny_i8(A, Bt, C, p->m, p->n, p->k, d->num_sms, stream) == cudaSuccess ? GEMM_OK
                                                                                               : GEMM_ERR_CUDA;
    }

    if (!tensor_map_encoder_available()) return GEMM_ERR_CUDA;
    uint16_t* Ah = reinterpret_cast<uint16_t*>(d->scratch);
    uint16_t* Bh = reinterpret_cast<uint16_t*>(d->scratch + round256(p->m * p->k_pitch * 2));
    // K split as in gemm_i8_run: the staging kernel zeroes C over the split tiles
    int64_t split_from = 0;
    StageZero z;
    const int split = tc_launch_split(C, p->m, p->n, p->k, p->bm, p->bn, p->grid, p->chunk_k / kTcBK, true,
                                      d->tc2_pairs, p->split_from == 0 ? p->split_k : 1, &split_from, &z);
    if (launch_stage_i8(A, Bt, Ah, Bh, p->m, p->n, p->k, p->k_pitch, z, d->err, d->num_sms, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    TcLaunch L;
    L.A16 = Ah;
    L.B16 = Bh;
    L.C = C;
    L.err = d->err;
    L.m = p->m;
    L.n = p->n;
    L.k = p->k;
    L.k_pitch = p->k_pitch;
    L.bm = p->bm;
    L.bn = p->bn;
    L.grid = p->grid;
    L.chunk_kb = p->chunk_k / kTcBK;
    L.int_out = true;
    L.split_k = split;
    L.split_from = split_from;
    const cudaError_t e = p->bm == 256 ? launch_tc2(L, d->tc2_pairs, stream) : launch_tc(L, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
