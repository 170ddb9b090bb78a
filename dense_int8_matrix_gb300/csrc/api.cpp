// C ABI of the library: argument checks, per-device state, workspace from a
// private stream-ordered pool, dispatch to the kernels, tracing.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/dense_int8_matrix.h"
#include "internal.h"

namespace gemm {
gemm_status make_plan(int32_t dtype, int64_t m, int64_t k, int64_t n, int32_t num_sms, gemm_plan* out);
}

using namespace gemm;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int* err_word = nullptr;
    int tc2_pairs = 0;                // co-resident CTA pairs of the two-SM kernel
    cudaMemPool_t pool = nullptr;
    // the blocked host entry point: side streams and events (created on first
    // use), taken by one call at a time
    cudaStream_t host_in = nullptr, host_stage = nullptr, host_gemm = nullptr, host_out = nullptr;
    std::vector<cudaEvent_t> host_events;
    std::mutex host_mu;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Per-device state, created on first use with that device current.
gemm_status device_state(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        s.num_sms = sms;
        s.supported = (major == 10 && minor == 3);
        if (s.supported) {
            if (device_error_word(&s.err_word) != cudaSuccess) return GEMM_ERR_CUDA;
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&s.pool, &props) != cudaSuccess) return GEMM_ERR_CUDA;
            uint64_t keep = UINT64_MAX;  // keep freed scratch for the next call
            if (cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess)
                return GEMM_ERR_CUDA;
            s.tc2_pairs = tc2_max_pairs();
        }
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

// ---------------------------------------------------------------- tracing --
// While tracing is on, every kernel launch is counted per kind, and every
// `every`-th run call ("sampled") records CUDA events around its launches.
struct TraceRec {
    int kind;
    cudaEvent_t start, stop;
};

std::mutex g_attr_mu;
struct AttrDone {
    const void* kern;
    int dev;
};
std::vector<AttrDone> g_attr_done;

std::mutex g_trace_mu;
bool g_trace_on = false;
int32_t g_trace_every = 1;
int64_t g_trace_calls = 0;
int32_t g_trace_launches[GEMM_KERNEL_KINDS] = {};
std::vector<TraceRec> g_trace;
size_t g_trace_used = 0;
size_t g_trace_cap = 0;   // units recorded at most in this trace (g_trace may hold more events)

// Whether this run call is sampled (decided once per call).
bool trace_sample_call() {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (!g_trace_on) return false;
    return (g_trace_calls++ % g_trace_every) == 0;
}

void trace_count(int kind) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (g_trace_on) ++g_trace_launches[kind];
}

// Events around the launches made in this scope, if the call is sampled.
struct TraceScope {
    TraceRec* rec = nullptr;
    cudaStream_t stream;
    TraceScope(int kind, cudaStream_t s, bool sampled) : stream(s) {
        if (!sampled) return;
        std::lock_guard<std::mutex> lock(g_trace_mu);
        if (g_trace_on && g_trace_used < g_trace_cap) {
            rec = &g_trace[g_trace_used++];
            rec->kind = kind;
            cudaEventRecord(rec->start, stream);
        }
    }
    ~TraceScope() {
        if (rec) cudaEventRecord(rec->stop, stream);
    }
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

gemm_status run_device(const gemm_plan* p, const void* A, const void* Bt, void* C, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    gemm_status st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (!tensor_map_encoder_available() && p->path == GEMM_PATH_TENSOR) return GEMM_ERR_CUDA;

    const bool sampled = trace_sample_call();
    if (p->path == GEMM_PATH_SKINNY) {
        if (skinny_tc_supported(p->m, p->n, p->k, A, Bt) && tensor_map_encoder_available()) {
            // The prologue writes an f16 copy of the small activation matrix
            // and zeroes C, which the tensor-core kernel adds its partial sums
            // into.  Both are launched with programmatic stream serialization
            // (each may start before the kernel in front of it ends), so the
            // two are timed as one unit.
            void* ws = nullptr;
            const size_t a_bytes = static_cast<size_t>(p->m * p->k * 2);
            if (cudaMallocFromPoolAsync(&ws, a_bytes, ds->pool, stream) != cudaSuccess) return GEMM_ERR_CUDA;
            cudaError_t e;
            {
                TraceScope t(GEMM_KERNEL_SKINNY, stream, sampled);
                e = launch_skinny_prologue(static_cast<const int8_t*>(A), static_cast<uint16_t*>(ws),
                                           static_cast<int32_t*>(C), p->m, p->n, p->k, ds->num_sms, stream);
                if (e == cudaSuccess) {
                    trace_count(GEMM_KERNEL_STAGE);
                    e = launch_skinny_tc(static_cast<const int8_t*>(Bt), static_cast<const uint16_t*>(ws),
                                         static_cast<int32_t*>(C), ds->err_word, p->m, p->n, p->k, ds->num_sms,
                                         stream);
                    if (e == cudaSuccess) trace_count(GEMM_KERNEL_SKINNY);
                }
            }
            cudaFreeAsync(ws, stream);
            return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
        }
        TraceScope t(GEMM_KERNEL_SKINNY, stream, sampled);
        if (launch_skinny_i8(static_cast<const int8_t*>(A), static_cast<const int8_t*>(Bt), static_cast<int32_t*>(C),
                             p->m, p->n, p->k, ds->num_sms, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        trace_count(GEMM_KERNEL_SKINNY);
        return GEMM_OK;
    }

    const bool is_i8 = p->dtype == GEMM_DTYPE_I8;
    const bool need_stage = is_i8 || (p->k_pitch != p->k);
    const int chunk_kb = p->chunk_k / kTcBK;

    // Tail split, recomputed for the tile and grid actually launched; the
    // staging kernel zeroes C over the split tiles, into which every slice adds.
    int64_t split_from = 0;
    StageZero z;
    const int split = tc_launch_split(static_cast<int32_t*>(C), p->m, p->n, p->k, p->bm, p->bn, p->grid, chunk_kb,
                                      is_i8, ds->tc2_pairs, p->split_from == 0 ? p->split_k : 1, &split_from, &z);
    const int64_t tiles = ((p->m + p->bm - 1) / p->bm) * ((p->n + p->bn - 1) / p->bn);

    void* ws = nullptr;
    const void* A16 = A;
    const void* B16 = Bt;
    // int8 A widened inside the two-SM kernel: only Bt is staged
    const bool a_on_chip = is_i8 && p->a_on_chip == 1;
    if (need_stage) {
        const int64_t a_bytes = a_on_chip ? 0 : ((p->m * p->k_pitch * 2 + 255) / 256) * 256;
        const int64_t b_bytes = ((p->n * p->k_pitch * 2 + 255) / 256) * 256;
        if (cudaMallocFromPoolAsync(&ws, static_cast<size_t>(a_bytes + b_bytes), ds->pool, stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        uint16_t* Ah = static_cast<uint16_t*>(ws);
        uint16_t* Bh = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + a_bytes);
        cudaError_t e;
        {
            TraceScope t(GEMM_KERNEL_STAGE, stream, sampled);
            if (a_on_chip)
                e = launch_stage_i8(static_cast<const int8_t*>(Bt), nullptr, Bh, nullptr, p->n, 0, p->k, p->k_pitch,
                                    z, ds->err_word, ds->num_sms, stream);
            else if (is_i8)
                e = launch_stage_i8(static_cast<const int8_t*>(A), static_cast<const int8_t*>(Bt), Ah, Bh, p->m, p->n,
                                    p->k, p->k_pitch, z, ds->err_word, ds->num_sms, stream);
            else
                e = launch_stage_b16(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(Bt), Ah, Bh, p->m,
                                     p->n, p->k, p->k_pitch, ds->num_sms, stream);
        }
        if (e != cudaSuccess) {
            cudaFreeAsync(ws, stream);
            return GEMM_ERR_CUDA;
        }
        trace_count(GEMM_KERNEL_STAGE);
        A16 = a_on_chip ? nullptr : Ah;
        B16 = Bh;
    }

    TcLaunch L;
    L.A8 = a_on_chip ? A : nullptr;
    L.A16 = A16;
    L.B16 = B16;
    L.C = C;
    L.err = ds->err_word;
    L.m = p->m;
    L.n = p->n;
    L.k = p->k;
    L.k_pitch = p->k_pitch;
    L.bm = p->bm;
    L.bn = p->bn;
    L.grid = p->grid;
    L.chunk_kb = chunk_kb;
    L.int_out = is_i8;
    // int8 problems are always staged, so the split tiles' C is zero
    L.split_k = need_stage ? split : 1;
    L.split_from = need_stage ? split_from : tiles;
    cudaError_t e;
    {
        TraceScope t(GEMM_KERNEL_TC, stream, sampled);
        e = p->bm == 256 ? launch_tc2(L, ds->tc2_pairs, stream) : launch_tc(L, stream);
    }
    if (e == cudaSuccess) trace_count(GEMM_KERNEL_TC);
    if (ws) cudaFreeAsync(ws, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Requantised output: D = q((float(C) * row_scale) * col_scale) with the exact
// int32 C never written to memory where a CTA completes it.  Whole tensor-path
// tiles are requantised in the GEMM's epilogue; the tiles of a K split add
// their int32 partial sums into pool scratch (zeroed by the staging kernel)
// and the requant kernel converts them afterwards; the skinny path adds into
// an int32 scratch C, which the requant kernel converts.
gemm_status run_requant(const gemm_plan* p, const int8_t* A, const int8_t* Bt, const float* rs, const float* cs,
                        int qmode, void* D, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    gemm_status st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (!tensor_map_encoder_available() && p->path == GEMM_PATH_TENSOR) return GEMM_ERR_CUDA;
    const int64_t m = p->m, n = p->n, k = p->k;
    auto al = [](int64_t b) { return static_cast<size_t>((b + 255) / 256 * 256); };
    RqOut o;
    o.D = D;
    o.row_scale = rs;
    o.col_scale = cs;
    o.ldd = n;
    o.qmode = qmode;
    const uintptr_t dp = reinterpret_cast<uintptr_t>(D);
    o.d_vec = qmode == kQuantBf16 ? ((dp % 16) == 0 && (n * 2) % 16 == 0) : ((dp % 8) == 0 && n % 8 == 0);
    const size_t c_bytes = al(m * n * 4);
    const bool sampled = trace_sample_call();

    if (p->path == GEMM_PATH_SKINNY) {
        const bool tc = skinny_tc_supported(m, n, k, A, Bt) && tensor_map_encoder_available();
        const size_t a16 = tc ? al(m * k * 2) : 0;
        void* ws = nullptr;
        if (cudaMallocFromPoolAsync(&ws, c_bytes + a16, ds->pool, stream) != cudaSuccess) return GEMM_ERR_CUDA;
        int32_t* C32 = static_cast<int32_t*>(ws);
        cudaError_t e;
        {
            TraceScope t(GEMM_KERNEL_SKINNY, stream, sampled);
            if (tc) {
                uint16_t* A16 = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + c_bytes);
                e = launch_skinny_prologue(A, A16, C32, m, n, k, ds->num_sms, stream);
                if (e == cudaSuccess) {
                    trace_count(GEMM_KERNEL_STAGE);
                    e = launch_skinny_tc(Bt, A16, C32, ds->err_word, m, n, k, ds->num_sms, stream);
                }
            } else {
                e = launch_skinny_i8(A, Bt, C32, m, n, k, ds->num_sms, stream);
            }
            if (e == cudaSuccess) trace_count(GEMM_KERNEL_SKINNY);
        }
        if (e == cudaSuccess) {
            TraceScope t(GEMM_KERNEL_REQUANT, stream, sampled);
            e = launch_requant(C32, n, o, m, n, RqTiles{}, ds->num_sms, stream);
            if (e == cudaSuccess) trace_count(GEMM_KERNEL_REQUANT);
        }
        cudaFreeAsync(ws, stream);
        return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    const int chunk_kb = p->chunk_k / kTcBK;
    int64_t split_from = 0;
    StageZero z;
    const int split = tc_launch_split(nullptr, m, n, k, p->bm, p->bn, p->grid, chunk_kb, true, ds->tc2_pairs,
                                      p->split_from == 0 ? p->split_k : 1, &split_from, &z);
    const int64_t tiles_m = (m + p->bm - 1) / p->bm, tiles_n = (n + p->bn - 1) / p->bn;
    const bool a_on_chip = p->a_on_chip == 1;   // int8 A widened inside the two-SM kernel
    const size_t a_bytes = a_on_chip ? 0 : al(m * p->k_pitch * 2), b_bytes = al(n * p->k_pitch * 2);
    const bool need_c = split > 1;   // int32 scratch for the split tiles' partial sums
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, a_bytes + b_bytes + (need_c ? c_bytes : 0), ds->pool, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    uint16_t* Ah = static_cast<uint16_t*>(ws);
    uint16_t* Bh = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + a_bytes);
    int32_t* C32 = need_c ? reinterpret_cast<int32_t*>(static_cast<char*>(ws) + a_bytes + b_bytes) : nullptr;
    z.C = C32;
    cudaError_t e;
    {
        TraceScope t(GEMM_KERNEL_STAGE, stream, sampled);
        e = a_on_chip ? launch_stage_i8(Bt, nullptr, Bh, nullptr, n, 0, k, p->k_pitch, z, ds->err_word, ds->num_sms,
                                        stream)
                      : launch_stage_i8(A, Bt, Ah, Bh, m, n, k, p->k_pitch, z, ds->err_word, ds->num_sms, stream);
    }
    if (e == cudaSuccess) {
        trace_count(GEMM_KERNEL_STAGE);
        TcLaunch L;
        L.A8 = a_on_chip ? A : nullptr;
        L.A16 = a_on_chip ? nullptr : Ah;
        L.B16 = Bh;
        L.C = C32;
        L.err = ds->err_word;
        L.m = m;
        L.n = n;
        L.k = k;
        L.k_pitch = p->k_pitch;
        L.bm = p->bm;
        L.bn = p->bn;
        L.grid = p->grid;
        L.chunk_kb = chunk_kb;
        L.int_out = true;
        L.split_k = split;
        L.split_from = split_from;
        L.rq = o;
        {
            TraceScope t(GEMM_KERNEL_TC, stream, sampled);
            e = p->bm == 256 ? launch_tc2(L, ds->tc2_pairs, stream) : launch_tc(L, stream);
        }
        if (e == cudaSuccess) trace_count(GEMM_KERNEL_TC);
    }
    if (e == cudaSuccess && need_c) {
        RqTiles tl;
        tl.bm = p->bm;
        tl.bn = p->bn;
        tl.tiles_m = static_cast<int>(tiles_m);
        tl.tiles_n = static_cast<int>(tiles_n);
        tl.tile_from = static_cast<int>(split_from);
        tl.tile_to = static_cast<int>(tiles_m * tiles_n);
        TraceScope t(GEMM_KERNEL_REQUANT, stream, sampled);
        e = launch_requant(C32, n, o, m, n, tl, ds->num_sms, stream);
        if (e == cudaSuccess) trace_count(GEMM_KERNEL_REQUANT);
    }
    cudaFreeAsync(ws, stream);
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// The end-to-end form is bound by the host link (about 200 GB/s each way on
// GB300, 256 GB/s both ways at once), above all by copying C back, so large
// tensor-path problems run as a pipeline on four streams: A is cut into row
// bands and Bt into column bands (rows of Bt); the bands go up one by one,
// each widened to f16 once on arrival, and every arrival completes a
// rectangle of C (the new row band against the column bands already up, or
// the new column band against the row bands already up), which one GEMM
// writes into the device copy of C and one strided copy brings down while
// later bands go up.  The bands go up in the order that completes the most
// of C per byte, so the download, the longest leg, starts after a small part
// of the input.  One GEMM per arrival (not per block): a GEMM takes at least
// one tile's K loop, so fewer, larger launches keep the GEMM stream ahead of
// the download.
// Bands: at least 1024 rows of A or of Bt each, at most 8 per matrix; only
// when C has at least 2048 rows and the copies move at least 32 MiB (a
// narrow C still gains: its GEMMs hide behind the upload of A).
constexpr int64_t kHostBandRows = 1024;
constexpr int64_t kHostMaxBands = 8;
constexpr int64_t kHostPipelineBytes = int64_t(32) << 20;

gemm_status host_streams(DeviceState* ds, size_t events) {
    if (!ds->host_out) {
        cudaStream_t s[4] = {nullptr, nullptr, nullptr, nullptr};
        for (auto& x : s)
            if (cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) != cudaSuccess) return GEMM_ERR_CUDA;
        ds->host_in = s[0];
        ds->host_stage = s[1];
        ds->host_gemm = s[2];
        ds->host_out = s[3];
    }
    while (ds->host_events.size() < events) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return GEMM_ERR_CUDA;
        ds->host_events.push_back(e);
    }
    return GEMM_OK;
}

// One rectangle of C on the tensor path, from operands already in device
// memory (16-bit, row pitch k_pitch); C is m x n with row pitch ldc and is
// written, not added to.  Rectangles run the two-SM 256 x 256 tile whatever
// their size: a launch lasts at least one tile's K loop, and on rectangles
// with fewer tiles than SMs the two-SM tile measured faster than the tiles
// the selector picks to fill every SM.  An int8 rectangle with fewer tiles
// than CTA pairs is split along K (whole 1024-element chunks) over the idle
// pairs, every slice adding into C zeroed just before.
gemm_status run_rect(DeviceState* ds, int32_t dtype, const void* A16, const void* B16, void* C, int64_t m, int64_t n,
                     int64_t ldc, int64_t k, int64_t k_pitch, bool sampled, cudaStream_t stream) {
    const bool is_i8 = dtype == GEMM_DTYPE_I8;
    const int pairs = ds->tc2_pairs > 0 ? ds->tc2_pairs : 1;
    const int64_t tiles = ((m + 255) / 256) * ((n + 255) / 256);
    const int64_t num_kb = (k + kTcBK - 1) / kTcBK;
    const int chunk_kb = is_i8 ? kI8ChunkK / kTcBK : static_cast<int>(num_kb);
    int split = 1;
    if (is_i8 && tiles < pairs) {
        const int64_t nchunks = (num_kb + chunk_kb - 1) / chunk_kb;
        int64_t s = pairs / tiles;
        if (s > nchunks) s = nchunks;
        if (s > kTcMaxSplit) s = kTcMaxSplit;
        split = static_cast<int>(s);
    }
    if (split > 1 && cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(n) * 4,
                                       static_cast<size_t>(m), stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    TcLaunch L;
    L.A16 = A16;
    L.B16 = B16;
    L.C = C;
    L.err = ds->err_word;
    L.m = m;
    L.n = n;
    L.k = k;
    L.k_pitch = k_pitch;
    L.bm = 256;
    L.bn = 256;
    L.grid = 2 * pairs;
    L.chunk_kb = chunk_kb;
    L.int_out = is_i8;
    L.split_k = split;
    L.split_from = split > 1 ? 0 : tiles;
    L.ldc = ldc;
    cudaError_t e;
    {
        TraceScope t(GEMM_KERNEL_TC, stream, sampled);
        e = launch_tc2(L, ds->tc2_pairs, stream);
    }
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    trace_count(GEMM_KERNEL_TC);
    return GEMM_OK;
}

gemm_status run_host_blocked(const gemm_plan* p, int32_t dtype, DeviceState* ds, const void* A, const void* Bt,
                             void* C, cudaStream_t stream, int64_t RM, int64_t RN) {
    const bool is_i8 = dtype == GEMM_DTYPE_I8;
    const size_t es = is_i8 ? 1 : 2;
    const int64_t m = p->m, n = p->n, k = p->k;
    const int64_t kp = p->k_pitch;
    const bool stage = is_i8 || kp != k;
    auto al = [](int64_t b) { return static_cast<size_t>((b + 255) / 256 * 256); };
    const size_t a_al = al(m * k * static_cast<int64_t>(es)), b_al = al(n * k * static_cast<int64_t>(es));
    const size_t a16_al = stage ? al(m * kp * 2) : 0, b16_al = stage ? al(n * kp * 2) : 0;
    const size_t c_bytes = static_cast<size_t>(m * n) * 4;

    std::lock_guard<std::mutex> lock(ds->host_mu);
    const size_t nev = 1 + 3 * static_cast<size_t>(RM + RN) + 4;
    gemm_status st = host_streams(ds, nev);
    if (st != GEMM_OK) return st;
    void* buf = nullptr;
    if (cudaMallocFromPoolAsync(&buf, a_al + b_al + a16_al + b16_al + c_bytes, ds->pool, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    char* dA = static_cast<char*>(buf);
    char* dB = dA + a_al;
    char* dA16 = dB + b_al;
    char* dB16 = dA16 + a16_al;
    char* dC = dB16 + b16_al;   // m x n, row pitch n, like the host's C
    const cudaStream_t s_in = ds->host_in, s_stage = ds->host_stage, s_gemm = ds->host_gemm, s_out = ds->host_out;
    cudaEvent_t* ev = ds->host_events.data();
    cudaEvent_t ev_start = ev[0];
    cudaEvent_t* ev_band = ev + 1;                 // [RM + RN]: per upload
    cudaEvent_t* ev_staged = ev + 1 + RM + RN;     // [RM + RN]: per band widened
    cudaEvent_t* ev_rect = ev + 1 + 2 * (RM + RN); // [RM + RN]: per rectangle of C
    cudaEvent_t ev_in_done = ev[nev - 4], ev_stage_done = ev[nev - 3], ev_gemm_done = ev[nev - 2],
                ev_out_done = ev[nev - 1];
    const bool sampled = trace_sample_call();
    auto edge = [](int64_t total, int64_t parts, int64_t i) { return total * i / parts; };

    // the side streams start after everything queued on `stream` (the pool
    // allocation included)
    if (cudaEventRecord(ev_start, stream) != cudaSuccess || cudaStreamWaitEvent(s_in, ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(s_stage, ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(s_gemm, ev_start, 0) != cudaSuccess || cudaStreamWaitEvent(s_out, ev_start, 0) != cudaSuccess)
        st = GEMM_ERR_CUDA;

    int64_t ia = 0, ib = 0;   // bands of A and of Bt up so far
    for (int64_t up = 0; st == GEMM_OK && up < RM + RN; ++up) {
        // next band: A's row band 0, Bt's column band 0, then whichever
        // completes more of C per byte uploaded (A on a tie)
        bool take_a;
        if (ia == 0 || ib == 0) {
            take_a = ia == 0;
        } else if (ia == RM || ib == RN) {
            take_a = ia < RM;
        } else {
            // an A band of r rows (r * k bytes) completes r x (columns up
            // so far) of C; a Bt band of r rows completes (rows up so far) x r
            take_a = edge(n, RN, ib) >= edge(m, RM, ia);
        }
        const int64_t idx = take_a ? ia : ib;
        const int64_t total = take_a ? m : n;
        const int64_t parts = take_a ? RM : RN;
        const int64_t r0 = edge(total, parts, idx), r1 = edge(total, parts, idx + 1);
        const char* h = static_cast<const char*>(take_a ? A : Bt) + static_cast<size_t>(r0 * k) * es;
        char* d = (take_a ? dA : dB) + static_cast<size_t>(r0 * k) * es;
        if (cudaMemcpyAsync(d, h, static_cast<size_t>((r1 - r0) * k) * es, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
            cudaEventRecord(ev_band[up], s_in) != cudaSuccess ||
            cudaStreamWaitEvent(stage ? s_stage : s_gemm, ev_band[up], 0) != cudaSuccess) {
            st = GEMM_ERR_CUDA;
            break;
        }
        // widening runs on its own stream, beside the multiplies of earlier
        // rectangles
        if (stage) {
            char* d16 = (take_a ? dA16 : dB16) + static_cast<size_t>(r0 * kp) * 2;
            cudaError_t e;
            {
                TraceScope t(GEMM_KERNEL_STAGE, s_stage, sampled);
                e = is_i8 ? launch_stage_i8(reinterpret_cast<const int8_t*>(d), nullptr, reinterpret_cast<uint16_t*>(d16),
                                            nullptr, r1 - r0, 0, k, kp, StageZero{}, ds->err_word, ds->num_sms, s_stage)
                          : launch_stage_b16(reinterpret_cast<const uint16_t*>(d), nullptr,
                                             reinterpret_cast<uint16_t*>(d16), nullptr, r1 - r0, 0, k, kp, ds->num_sms,
                                             s_stage);
            }
            if (e != cudaSuccess || cudaEventRecord(ev_staged[up], s_stage) != cudaSuccess ||
                cudaStreamWaitEvent(s_gemm, ev_staged[up], 0) != cudaSuccess) {
                st = GEMM_ERR_CUDA;
                break;
            }
            trace_count(GEMM_KERNEL_STAGE);
        }
        if (take_a)
            ++ia;
        else
            ++ib;
        // the rectangle this band completes
        const int64_t m0 = take_a ? r0 : 0, m1 = take_a ? r1 : edge(m, RM, ia);
        const int64_t n0 = take_a ? 0 : r0, n1 = take_a ? edge(n, RN, ib) : r1;
        if (m1 <= m0 || n1 <= n0) continue;
        const size_t a_off = stage ? static_cast<size_t>(m0 * kp) * 2 : static_cast<size_t>(m0 * k) * es;
        const size_t b_off = stage ? static_cast<size_t>(n0 * kp) * 2 : static_cast<size_t>(n0 * k) * es;
        const char* opA = (stage ? dA16 : dA) + a_off;
        const char* opB = (stage ? dB16 : dB) + b_off;
        const size_t c_off = static_cast<size_t>(m0 * n + n0) * 4;
        st = run_rect(ds, dtype, opA, opB, dC + c_off, m1 - m0, n1 - n0, n, k, stage ? kp : k, sampled, s_gemm);
        if (st == GEMM_OK &&
            (cudaEventRecord(ev_rect[up], s_gemm) != cudaSuccess || cudaStreamWaitEvent(s_out, ev_rect[up], 0) != cudaSuccess ||
             cudaMemcpy2DAsync(static_cast<char*>(C) + c_off, static_cast<size_t>(n) * 4, dC + c_off,
                               static_cast<size_t>(n) * 4, static_cast<size_t>(n1 - n0) * 4,
                               static_cast<size_t>(m1 - m0), cudaMemcpyDeviceToHost, s_out) != cudaSuccess))
            st = GEMM_ERR_CUDA;
    }
    // `stream` (and the pool's free below) waits for all four streams,
    // whatever was queued before an error
    cudaEventRecord(ev_in_done, s_in);
    cudaEventRecord(ev_stage_done, s_stage);
    cudaEventRecord(ev_gemm_done, s_gemm);
    cudaEventRecord(ev_out_done, s_out);
    cudaStreamWaitEvent(stream, ev_in_done, 0);
    cudaStreamWaitEvent(stream, ev_stage_done, 0);
    cudaStreamWaitEvent(stream, ev_gemm_done, 0);
    cudaStreamWaitEvent(stream, ev_out_done, 0);
    cudaFreeAsync(buf, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess && st == GEMM_OK) st = GEMM_ERR_CUDA;
    return st;
}

gemm_status run_host(const gemm_plan* p, int32_t dtype, const void* A, const void* Bt, void* C, cudaStream_t stream) {
    gemm_status st = check_plan(p, dtype);
    if (st != GEMM_OK) return st;
    if (!A || !Bt || !C) return GEMM_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    const size_t es = dtype == GEMM_DTYPE_I8 ? 1 : 2;
    const size_t a_bytes = static_cast<size_t>(p->m * p->k) * es;
    const size_t b_bytes = static_cast<size_t>(p->n * p->k) * es;
    const size_t c_bytes = static_cast<size_t>(p->m * p->n) * 4;
    if (p->path == GEMM_PATH_TENSOR && static_cast<int64_t>(a_bytes + b_bytes + c_bytes) >= kHostPipelineBytes &&
        p->m >= 2 * kHostBandRows) {
        int64_t RM = p->m / kHostBandRows, RN = p->n / kHostBandRows;
        if (RM > kHostMaxBands) RM = kHostMaxBands;
        if (RN > kHostMaxBands) RN = kHostMaxBands;
        if (RN < 1) RN = 1;
        return run_host_blocked(p, dtype, ds, A, Bt, C, stream, RM, RN);
    }
    const size_t a_al = (a_bytes + 255) / 256 * 256, b_al = (b_bytes + 255) / 256 * 256;
    void* buf = nullptr;
    if (cudaMallocFromPoolAsync(&buf, a_al + b_al + c_bytes, ds->pool, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    char* dA = static_cast<char*>(buf);
    char* dB = dA + a_al;
    char* dC = dB + b_al;
    if (cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(dB, Bt, b_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        st = GEMM_ERR_CUDA;
    if (st == GEMM_OK) st = run_device(p, dA, dB, dC, stream);
    if (st == GEMM_OK && cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        st = GEMM_ERR_CUDA;
    cudaFreeAsync(buf, stream);
    if (cudaStreamSynchronize(stream) != cudaSuccess && st == GEMM_OK) st = GEMM_ERR_CUDA;
    return st;
}

}  // namespace

// Argument checks shared with the allocation-free entry point (noalloc.cu).
gemm_status gemm::check_plan(const gemm_plan* p, int32_t dtype) {
    if (!p || p->version != GEMM_PLAN_VERSION || p->dtype != dtype) return GEMM_ERR_INVALID_ARG;
    if (p->m < 1 || p->k < 1 || p->n < 1) return GEMM_ERR_INVALID_ARG;
    if (p->path == GEMM_PATH_SKINNY) {
        if (dtype != GEMM_DTYPE_I8 || p->m > 128 || p->grid < 1) return GEMM_ERR_INVALID_ARG;
        return GEMM_OK;
    }
    if (p->path != GEMM_PATH_TENSOR) return GEMM_ERR_INVALID_ARG;
    // a plan may be edited to force a tile, but only to one that is compiled
    if (p->bm == 256) {
        if (p->bn != 256 || (p->grid % 2) != 0) return GEMM_ERR_INVALID_ARG;
    } else {
        if (p->bm != 64 && p->bm != 128) return GEMM_ERR_INVALID_ARG;
        if (p->bn != 32 && p->bn != 64 && p->bn != 128 && p->bn != 256) return GEMM_ERR_INVALID_ARG;
    }
    if (p->grid < 1 || p->k_pitch < p->k || (p->k_pitch % 8) != 0 || p->chunk_k < kTcBK ||
        (p->chunk_k % kTcBK) != 0)
        return GEMM_ERR_INVALID_ARG;
    if (dtype == GEMM_DTYPE_I8 && p->chunk_k > kI8ChunkK) return GEMM_ERR_INVALID_ARG;
    if (p->split_k < 1 || p->split_k > kTcMaxSplit) return GEMM_ERR_INVALID_ARG;
    // A widened on chip: the two-SM kernel, int8, a 16-byte row pitch of int8 A
    if (p->a_on_chip != 0 && (p->a_on_chip != 1 || dtype != GEMM_DTYPE_I8 || p->bm != 256 || (p->k % 16) != 0))
        return GEMM_ERR_INVALID_ARG;
    // bf16 problems accumulate the whole K in one TMEM chunk
    if (dtype == GEMM_DTYPE_BF16 && p->chunk_k < p->k) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

gemm_status gemm::check_ptrs(const void* A, const void* Bt, const void* C) {
    if (!A || !Bt || !C) return GEMM_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Bt, 16) || !aligned(C, 4)) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

cudaError_t gemm::kernel_attrs_once(const void* kern, int smem_bytes, bool max_carveout) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    for (const AttrDone& d : g_attr_done)
        if (d.kern == kern && d.dev == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess) g_attr_done.push_back(AttrDone{kern, dev});
    return e;
}

extern "C" {

gemm_status gemm_plan_for_sms(int32_t dtype, int64_t m, int64_t k, int64_t n, int32_t num_sms, gemm_plan* out) {
    return make_plan(dtype, m, k, n, num_sms, out);
}

static gemm_status plan_current(int32_t dtype, int64_t m, int64_t k, int64_t n, gemm_plan* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    // argument errors first, without touching the device
    gemm_plan probe;
    gemm_status st = make_plan(dtype, m, k, n, 148, &probe);
    if (st != GEMM_OK) return st;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != GEMM_OK) return st;
    return make_plan(dtype, m, k, n, ds->num_sms, out);
}

gemm_status gemm_i8_plan(int64_t m, int64_t k, int64_t n, gemm_plan* out) {
    return plan_current(GEMM_DTYPE_I8, m, k, n, out);
}

gemm_status gemm_bf16_plan(int64_t m, int64_t k, int64_t n, gemm_plan* out) {
    return plan_current(GEMM_DTYPE_BF16, m, k, n, out);
}

gemm_status gemm_i8_run(const gemm_plan* plan, const int8_t* A, const int8_t* Bt, int32_t* C, void* stream) {
    gemm_status st = check_plan(plan, GEMM_DTYPE_I8);
    if (st != GEMM_OK) return st;
    st = check_ptrs(A, Bt, C);
    if (st != GEMM_OK) return st;
    return run_device(plan, A, Bt, C, static_cast<cudaStream_t>(stream));
}

gemm_status gemm_bf16_run(const gemm_plan* plan, const uint16_t* A, const uint16_t* Bt, float* C, void* stream) {
    gemm_status st = check_plan(plan, GEMM_DTYPE_BF16);
    if (st != GEMM_OK) return st;
    st = check_ptrs(A, Bt, C);
    if (st != GEMM_OK) return st;
    return run_device(plan, A, Bt, C, static_cast<cudaStream_t>(stream));
}

gemm_status gemm_i8_run_requant(const gemm_plan* plan, const int8_t* A, const int8_t* Bt, const float* row_scale,
                                const float* col_scale, int32_t out_type, void* D, void* stream) {
    gemm_status st = check_plan(plan, GEMM_DTYPE_I8);
    if (st != GEMM_OK) return st;
    if (out_type != GEMM_OUT_BF16 && out_type != GEMM_OUT_I8) return GEMM_ERR_INVALID_ARG;
    if (!A || !Bt || !D || !row_scale || !col_scale) return GEMM_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Bt, 16) || !aligned(row_scale, 16) || !aligned(col_scale, 16) ||
        (out_type == GEMM_OUT_BF16 && !aligned(D, 2)))
        return GEMM_ERR_MISALIGNED;
    return run_requant(plan, A, Bt, row_scale, col_scale, out_type == GEMM_OUT_BF16 ? kQuantBf16 : kQuantI8, D,
                       static_cast<cudaStream_t>(stream));
}

gemm_status gemm_i8_run_host(const gemm_plan* plan, const int8_t* A, const int8_t* Bt, int32_t* C, void* stream) {
    return run_host(plan, GEMM_DTYPE_I8, A, Bt, C, static_cast<cudaStream_t>(stream));
}

gemm_status gemm_bf16_run_host(const gemm_plan* plan, const uint16_t* A, const uint16_t* Bt, float* C,
                               void* stream) {
    return run_host(plan, GEMM_DTYPE_BF16, A, Bt, C, static_cast<cudaStream_t>(stream));
}

gemm_status gemm_device_error(void* stream, int32_t* code) {
    if (code) *code = 0;
    DeviceState* ds = nullptr;
    gemm_status st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ds->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (v == 0) return GEMM_OK;
    if (code) *code = v;
    if (cudaMemset(ds->err_word, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_ERR_TIMEOUT;
}

gemm_status gemm_pool_usage(int64_t* reserved_bytes, int64_t* used_high_bytes, int32_t reset_high) {
    if (!reserved_bytes || !used_high_bytes) return GEMM_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    gemm_status st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    uint64_t reserved = 0, high = 0;
    if (cudaMemPoolGetAttribute(ds->pool, cudaMemPoolAttrReservedMemCurrent, &reserved) != cudaSuccess ||
        cudaMemPoolGetAttribute(ds->pool, cudaMemPoolAttrUsedMemHigh, &high) != cudaSuccess)
        return GEMM_ERR_CUDA;
    *reserved_bytes = static_cast<int64_t>(reserved);
    *used_high_bytes = static_cast<int64_t>(high);
    if (reset_high) {
        uint64_t zero = 0;   // the high-water mark restarts from the current use
        if (cudaMemPoolSetAttribute(ds->pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

gemm_status gemm_trace_begin(int32_t capacity, int32_t every) {
    if (capacity < 0 || every < 1) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    while (g_trace.size() < static_cast<size_t>(capacity)) {
        TraceRec r;
        r.kind = 0;
        if (cudaEventCreate(&r.start) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaEventCreate(&r.stop) != cudaSuccess) {
            cudaEventDestroy(r.start);
            return GEMM_ERR_CUDA;
        }
        g_trace.push_back(r);
    }
    g_trace_used = 0;
    g_trace_cap = static_cast<size_t>(capacity);
    g_trace_every = every;
    g_trace_calls = 0;
    for (int i = 0; i < GEMM_KERNEL_KINDS; ++i) g_trace_launches[i] = 0;
    g_trace_on = true;
    return GEMM_OK;
}

gemm_status gemm_trace_collect(float* ms_per_kind, int32_t* timed_per_kind, int32_t* launches_per_kind) {
    if (!ms_per_kind || !timed_per_kind || !launches_per_kind) return GEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    for (int i = 0; i < GEMM_KERNEL_KINDS; ++i) {
        ms_per_kind[i] = 0.f;
        timed_per_kind[i] = 0;
        launches_per_kind[i] = g_trace_launches[i];
    }
    gemm_status st = GEMM_OK;
    for (size_t i = 0; i < g_trace_used; ++i) {
        TraceRec& r = g_trace[i];
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
            st = GEMM_ERR_CUDA;
            continue;
        }
        if (r.kind >= 0 && r.kind < GEMM_KERNEL_KINDS) {
            ms_per_kind[r.kind] += ms;
            timed_per_kind[r.kind] += 1;
        }
    }
    g_trace_on = false;
    g_trace_used = 0;
    return st;
}

gemm_status gemm_tc_kernel_info(int32_t bm, int32_t bn, int32_t dtype, int32_t* regs, int32_t* ctas_per_sm) {
    if (!regs || !ctas_per_sm) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_DTYPE_I8 && dtype != GEMM_DTYPE_BF16) return GEMM_ERR_INVALID_ARG;
    if (bm == 256 && bn == 256) {
        *regs = tc2_num_regs(dtype == GEMM_DTYPE_I8);
        *ctas_per_sm = *regs > 0 ? 1 : 0;
    } else {
        *regs = tc_num_regs(bm, bn, dtype == GEMM_DTYPE_I8);
        *ctas_per_sm = tc_occupancy(bm, bn, dtype == GEMM_DTYPE_I8);
    }
    return *regs < 0 ? GEMM_ERR_INVALID_ARG : GEMM_OK;
}

gemm_status gemm_selftest_wait_timeout(int32_t timeout_us, void* stream) {
    if (timeout_us < 1 || timeout_us > 2000000) return GEMM_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    gemm_status st = device_state(&ds);
    if (st != GEMM_OK) return st;
    if (!ds->supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (launch_selftest_wait(ds->err_word, static_cast<uint64_t>(timeout_us) * 1000u,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_OVERFLOW_RISK: return "GEMM_ERR_OVERFLOW_RISK";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    }
    return "GEMM_ERR_UNKNOWN";
}

}  // extern "C"
