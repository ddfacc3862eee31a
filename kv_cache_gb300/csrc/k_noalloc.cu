// kvring_attend_noalloc: the attention call over a cache the caller holds,
// using no device memory beyond what the caller passes in and one fixed
// scratch array that lives in this file.
//
// Who needs it: callers whose device memory is all handed out up front by
// their own arena or pool and who may not call cudaMalloc/cudaFree (or any
// allocating library routine, torch's caching allocator included) while they
// serve -- for instance an engine that owns a fixed slab of HBM and places the
// FP8 cache in it itself.  kvring_create allocates the rings and its scratch;
// this entry point allocates nothing.
//
// The only intermediate the attention needs here is the e4m3 copy of Q (and
// each row's amax), written by the Q-prep kernel and read by the attention
// kernel through TMA.  It lives in g_noalloc_scratch below, a file-scope
// __device__ array of fixed size: every GPU that loads this library holds it
// (2.06 MB) until the process exits.  KV splits, when the call has them, merge
// as thread-block clusters through distributed shared memory, so no split
// partials or counters are needed either.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

#include "kvring_internal.h"

namespace kvring_impl {

// Scratch capacity in (head, padded query row) pairs: 16,384 rows, e.g. 16 heads
// x 1,024 queries or 64 heads x 256 queries.  Query rows are padded to a
// multiple of 256 (pairs of 128-row tiles).
constexpr int kNoAllocMaxRows = 16384;
constexpr size_t kNoAllocQBytes = (size_t)kNoAllocMaxRows * 128;           // e4m3 Q rows, d <= 128
constexpr size_t kNoAllocAmaxOff = kNoAllocQBytes;                         // float per row
constexpr size_t kNoAllocErrOff = kNoAllocAmaxOff + kNoAllocMaxRows * 4;   // spare error word (4 ints)
constexpr size_t kNoAllocBytes = kNoAllocErrOff + 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_dev[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int g_num_sms[kMaxDevices] = {};
int g_cluster_cap[kMaxDevices][2][5] = {};  // [device][d = 64, 128][splits 2..4]: attention clusters held at once

int noalloc_fail(int code, const std::string& msg) {
    set_thread_error("kvring_attend_noalloc: " + msg);
    return code;
}

// Device address of the scratch array on the current device, and the device's
// SM count and attention cluster capacities.  The host-side symbol
// g_noalloc_scratch is only a stand-in and must never be handed to a kernel; the
// address comes from cudaGetSymbolAddress, once per device, with that device
// current.
int scratch_address(int dev, uint8_t** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return noalloc_fail(KVRING_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || sms < 1)
            return noalloc_fail(KVRING_ECUDA, std::string("multiprocessor count: ") + cudaGetErrorString(e));
        for (int di = 0; di < 2; ++di)
            for (int sp = 2; sp <= 4; ++sp) g_cluster_cap[dev][di][sp] = attend_max_clusters(di ? 128 : 64, sp);
        g_num_sms[dev] = sms;
        g_scratch_dev[dev] = static_cast<uint8_t*>(ptr);
    }
    *out = g_scratch_dev[dev];
    return KVRING_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace kvring_impl

using namespace kvring_impl;

extern "C" int kvring_attend_noalloc(const void* k8, const void* vt8, const float* kamax, const float* vamax,
                                     const float* rope, int64_t rope_rows, int64_t q_pos0, const void* q_bf16, int32_t n_q,
                                     int32_t num_heads, int32_t head_dim, int32_t slots_padded, int32_t count,
                                     float* out_f32, int* err_word, void* cuda_stream) {
    if (n_q == 0) return KVRING_OK;
    if (!k8 || !vt8 || !kamax || !vamax || !rope || !q_bf16 || !out_f32)
        return noalloc_fail(KVRING_EINVAL, "a required pointer is NULL");
    if (head_dim != 64 && head_dim != 128) return noalloc_fail(KVRING_EINVAL, "head_dim must be 64 or 128");
    if (num_heads < 1 || num_heads > 256) return noalloc_fail(KVRING_EINVAL, "num_heads out of range [1, 256]");
    if (slots_padded < 128 || slots_padded % 128 != 0)
        return noalloc_fail(KVRING_EINVAL, "slots_padded must be a positive multiple of 128");
    if (count < 1 || count > slots_padded) return noalloc_fail(KVRING_EINVAL, "count out of range [1, slots_padded]");
    if (n_q < 0 || q_pos0 < 0) return noalloc_fail(KVRING_EINVAL, "n_q and q_pos0 must be >= 0");
    // Q prep reads rope rows q_pos0 .. q_pos0 + n_q - 1
    if (rope_rows < 1 || q_pos0 > rope_rows - (int64_t)n_q)
        return noalloc_fail(KVRING_EINVAL, "rope has " + std::to_string(rope_rows) + " rows; the queries need rows up to " +
                                               std::to_string(q_pos0 + n_q - 1));
    const int64_t tstride = ((int64_t)n_q + 255) / 256 * 256;
    if ((int64_t)num_heads * tstride > kNoAllocMaxRows)
        return noalloc_fail(KVRING_EINVAL, "num_heads x n_q (padded to 256) = " + std::to_string(num_heads * tstride) +
                                               " exceeds the fixed scratch of " + std::to_string(kNoAllocMaxRows) +
                                               " rows; use kvring_attend or split the heads");
    if (!aligned(k8, 16) || !aligned(vt8, 16) || !aligned(q_bf16, 16) || !aligned(out_f32, 16) ||
        !aligned(kamax, 16) || !aligned(vamax, 16) || !aligned(rope, 8) || (err_word && !aligned(err_word, 4)))
        return noalloc_fail(KVRING_EINVAL, "k8, vt8, kamax, vamax, q and out must be 16-byte aligned (rope 8)");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(KVRING_ENODEV, std::string("no CUDA device: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(KVRING_ENODEV, "device index out of range");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major * 10 + minor != 103) return noalloc_fail(KVRING_ENODEV, "this library is built for sm_103a");
    uint8_t* scratch = nullptr;
    int rc = scratch_address(dev, &scratch);
    if (rc) return rc;

    const int H = num_heads, d = head_dim;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    uint8_t* q8 = scratch;
    float* qamax = reinterpret_cast<float*>(scratch + kNoAllocAmaxOff);
    int* err = err_word ? err_word : reinterpret_cast<int*>(scratch + kNoAllocErrOff);
    // The library's own word (err_word NULL) starts every call at zero, so a
    // time-out of an earlier call never masks one of this call; a caller's word
    // is left as it is (it keeps the first time-out until the caller clears it).
    if (!err_word) {
        e = cudaMemsetAsync(err, 0, 4 * sizeof(int), s);
        if (e != cudaSuccess) return noalloc_fail(KVRING_ECUDA, std::string("clearing the error word: ") + cudaGetErrorString(e));
    }

    // Q prep writes every row of the Q scratch it uses (pad rows as zeros), so
    // nothing left by an earlier call is read.
    QPrepParams qp{};
    qp.q = static_cast<const uint16_t*>(q_bf16);
    qp.q8 = q8;
    qp.qamax = qamax;
    qp.rope = reinterpret_cast<const float2*>(rope);
    qp.pos0 = q_pos0;
    qp.T = n_q;
    qp.Tpad = (n_q + 127) / 128 * 128;
    qp.H = H;
    qp.d = d;
    qp.Tstride = (int)tstride;

    AttendMaps maps{};
    const CUtensorMapSwizzle swz_d = d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const cuuint64_t kdims[3] = {(cuuint64_t)d, (cuuint64_t)slots_padded, (cuuint64_t)H};
    const cuuint64_t kstr[2] = {(cuuint64_t)d, (cuuint64_t)slots_padded * d};
    const cuuint32_t kbox[3] = {(cuuint32_t)d, 128, 1};
    const cuuint64_t vdims[3] = {(cuuint64_t)slots_padded, (cuuint64_t)d, (cuuint64_t)H};
    const cuuint64_t vstr[2] = {(cuuint64_t)slots_padded, (cuuint64_t)slots_padded * d};
    const cuuint32_t vbox[3] = {128, (cuuint32_t)d, 1};
    const cuuint64_t qdims[3] = {(cuuint64_t)d, (cuuint64_t)tstride, (cuuint64_t)H};
    const cuuint64_t qstr[2] = {(cuuint64_t)d, (cuuint64_t)tstride * d};
    const cuuint32_t qbox[3] = {(cuuint32_t)d, 128, 1};
    if ((rc = encode_u8_map(&maps.k8, const_cast<void*>(k8), kdims, kstr, kbox, swz_d)) ||
        (rc = encode_u8_map(&maps.vt8, const_cast<void*>(vt8), vdims, vstr, vbox, CU_TENSOR_MAP_SWIZZLE_128B)) ||
        (rc = encode_u8_map(&maps.q8, q8, qdims, qstr, qbox, swz_d)))
        return noalloc_fail(rc, "tensor map encoding failed");

    AttendParams ap{};
    ap.kamax = kamax;
    ap.vamax = vamax;
    ap.qamax = qamax;
    ap.out = out_f32;
    ap.part_o = nullptr;       // one KV split: the kernel writes O straight to out
    ap.part_ml = nullptr;
    ap.counters = nullptr;
    ap.err = err;
    ap.T = n_q;
    ap.H = H;
    ap.d = d;
    ap.Rpad = slots_padded;
    ap.Tstride = (int)tstride;
    ap.count = count;
    ap.layer = 0;
    ap.npairs = (n_q + 255) / 256;
    ap.ntiles = (count + 127) / 128;
    // KV splits: as many as keep every CTA in one wave and every cluster of them
    // on the device at once (fewest tile-times per CTA; one split otherwise)
    const int units = H * ap.npairs;
    int best_se = 1, best_tps = ap.ntiles;
    long long best_cost = -1;
    for (int sp = 1; sp <= std::min(4, ap.ntiles); ++sp) {
        const int tps = (ap.ntiles + sp - 1) / sp;
        const int se = (ap.ntiles + tps - 1) / tps;
        if (se > 1 && g_cluster_cap[dev][d == 128 ? 1 : 0][se] < units) continue;
        const long long waves = ((long long)units * se + g_num_sms[dev] - 1) / g_num_sms[dev];
        const long long cost = waves * tps;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_se = se; best_tps = tps; }
    }
    ap.splits = best_se;
    ap.tiles_per_split = best_tps;
    ap.log2e_rsqrt_d = (float)(1.4426950408889634 / std::sqrt((double)d));
    ap.timeout_ns = 2000000000LL;
    ap.skip_tile = -1;
    ap.coop = 0;
    ap.cluster = best_se > 1 ? 1 : 0;

    e = launch_qprep(qp, s);
    if (e == cudaSuccess) e = launch_attend(ap, maps, s);
    if (e != cudaSuccess) return noalloc_fail(KVRING_ECUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
    return KVRING_OK;
}
