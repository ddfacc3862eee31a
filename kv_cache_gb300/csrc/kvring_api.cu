// Host side of the C ABI: argument checks, ring bookkeeping, device buffers,
// TMA tensor maps and kernel launches.  See include/kvring.h for the contract.
//
// Bookkeeping follows the pages' ring buffer (ai.info, "Characters funziona in
// tempo reale su quattro H100", section "La gestione della cache spostata al
// momento della scrittura"): token j of a chunk goes to slot (head + j) mod R at
// position next_pos + j; the window advances by overwriting, never by copying;
// a position reset subtracts delta = next_pos - count from every position.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "kvring_internal.h"

using namespace kvring_impl;

namespace {

struct LayerState {
    int64_t head = 0, count = 0, next_pos = 0, writes = 0, last_pos = 0, last_n = 0;
    int cur = 0;                  // naive upkeep: which window buffer holds the window
    bool fresh = false;           // naive upkeep: FP8 cache refreshed since the last change
    std::vector<int32_t> pos;     // [R], -1 = empty
    std::vector<int32_t> chunk;   // [R], -1 = empty
};

thread_local std::string g_create_error;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

struct kvring {
    kvring_config cfg{};
    bool host_only = false;
    bool naive = false;         // KVRING_FLAG_NAIVE_UPKEEP
    bool rope3d = false;        // KVRING_FLAG_ROPE_3D
    int device = 0, num_sms = 0;
    int64_t Rpad = 0, Tstride = 0;
    int max_splits = 1;
    int cluster_cap[5] = {0, 0, 0, 0, 0};   // per split count (2-4): attention clusters the device holds at once
    int64_t resets = 0;
    std::vector<LayerState> layers;
    // device buffers (owned)
    uint8_t* k8 = nullptr;      // [L][H][Rpad][d]
    uint8_t* vt8 = nullptr;     // [L][H][d][Rpad]
    float* kamax = nullptr;     // [L][H][Rpad]
    float* vamax = nullptr;     // [L][H][Rpad]
    float2* rope = nullptr;     // [max_position][d/2]
    uint8_t* q8 = nullptr;      // [H][Tstride][d]
    float* qamax = nullptr;     // [H][Tstride]
    float* part_o = nullptr;    // [max_splits][H][Tstride][d]
    float* part_ml = nullptr;   // [max_splits][H][Tstride][2]
    int* counters = nullptr;    // [2][H][Tstride/256] split arrivals (and merges done) per (head, query pair)
    float* wpart = nullptr;     // [2][amax blocks][H] per-block amax partials of the write kernels
    uint16_t* kwin = nullptr;   // naive upkeep: bf16 windows [2 buffers][L][H][Rpad][d]
    uint16_t* vwin = nullptr;
    float* kaw = nullptr;       // naive upkeep: chunk amax of each window row [2][L][H][Rpad]
    float* vaw = nullptr;
    int* err = nullptr;         // [4]
    AttendMaps maps{};
    CUtensorMap rope_map{};     // the RoPE table for the write kernel
    // testing aid
    uint64_t launches = 0;
    int debug_skip_tile = -1;
    int debug_skip_group = -1;          // testing aid for the write kernel's waits
    long long debug_write_timeout_ns = 0;
    int last_q_rows = 0;        // query rows of the latest attention call (for kvring_snapshot_q)
    long long debug_timeout_ns = 0;
    std::string error;
};

namespace {

int fail(kvring_t* r, int code, const std::string& msg) {
    if (r) r->error = msg; else g_create_error = msg;
    return code;
}

int cuda_fail(kvring_t* r, cudaError_t e, const char* what) {
    return fail(r, KVRING_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

void free_device(kvring_t* r) {
    void* ptrs[] = {r->k8, r->vt8, r->kamax, r->vamax, r->rope, r->q8, r->qamax, r->part_o, r->part_ml, r->counters,
                    r->wpart, r->kwin, r->vwin, r->kaw, r->vaw, r->err};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    r->k8 = r->vt8 = r->q8 = nullptr;
    r->kamax = r->vamax = r->qamax = r->part_o = r->part_ml = nullptr;
    r->rope = nullptr;
    r->counters = nullptr;
    r->wpart = nullptr;
    r->kwin = r->vwin = nullptr;
    r->kaw = r->vaw = nullptr;
    r->err = nullptr;
}

// Angles p * w_i formed and evaluated in float64 (w_i = theta^(-2i/d)), cos and
// sin rounded once to float32; one row of d/2 (cos, sin) pairs per position.
// 3-D video layout (KVRING_FLAG_ROPE_3D): running index p = frame * S + s has
// coordinates t = p / S, h = s / W, w = s % W; pairs [0, pt) turn by t, the next
// ph by h, the rest by w, each band with the frequencies of its own width.
struct Rope3D {
    int S, W, pt, ph;
};

void build_rope_table(std::vector<float2>& tab, int max_pos, int d, double theta, const Rope3D* r3) {
    const int half = d / 2;
    std::vector<double> w(half);
    std::vector<int> band(half, 0);   // 3-D: 0 = time, 1 = height, 2 = width
    if (!r3) {
        for (int i = 0; i < half; ++i) w[i] = std::pow(theta, -2.0 * i / d);
    } else {
        const int n[3] = {r3->pt, r3->ph, half - r3->pt - r3->ph};
        int i = 0;
        for (int b = 0; b < 3; ++b)
            for (int k = 0; k < n[b]; ++k, ++i) {
                w[i] = std::pow(theta, -2.0 * k / (2 * n[b]));
                band[i] = b;
            }
    }
    tab.resize((size_t)max_pos * half);
    unsigned nth = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    std::vector<std::thread> th;
    for (unsigned k = 0; k < nth; ++k) {
        th.emplace_back([&, k] {
            for (int64_t p = k; p < max_pos; p += nth)
                for (int i = 0; i < half; ++i) {
                    int64_t coord = p;
                    if (r3) {
                        const int64_t s = p % r3->S;
                        coord = band[i] == 0 ? p / r3->S : band[i] == 1 ? s / r3->W : s % r3->W;
                    }
                    const double ang = (double)coord * w[i];
                    tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
                }
        });
    }
    for (auto& t : th) t.join();
}

int make_map(kvring_t* r, CUtensorMap* map, void* base, const cuuint64_t dims[3], const cuuint64_t strides[2],
             const cuuint32_t box[3], CUtensorMapSwizzle swz) {
    const int rc = kvring_impl::encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, swz);
    if (rc) return fail(r, rc, "cuTensorMapEncodeTiled failed");
    return KVRING_OK;
}

int check_config(const kvring_config* c) {
    if (!c) return fail(nullptr, KVRING_EINVAL, "config is NULL");
    if (c->num_layers < 1 || c->num_layers > KVRING_MAX_LAYERS) return fail(nullptr, KVRING_EINVAL, "num_layers out of range [1, 256]");
    if (c->num_heads < 1 || c->num_heads > 256) return fail(nullptr, KVRING_EINVAL, "num_heads out of range [1, 256]");
    if (c->head_dim != 64 && c->head_dim != 128) return fail(nullptr, KVRING_EINVAL, "head_dim must be 64 or 128");
    if (c->capacity < 1 || c->capacity > (1 << 20)) return fail(nullptr, KVRING_EINVAL, "capacity out of range [1, 2^20]");
    if (c->max_tokens_per_write < 1 || c->max_tokens_per_write > c->capacity || c->max_tokens_per_write > 2048)
        return fail(nullptr, KVRING_EINVAL, "max_tokens_per_write out of range [1, min(capacity, 2048)]");
    if (c->max_position < 0) return fail(nullptr, KVRING_EINVAL, "max_position must be >= 0");
    if (c->rope_theta < 0 || !std::isfinite(c->rope_theta)) return fail(nullptr, KVRING_EINVAL, "rope_theta must be finite and >= 0");
    if (c->flags & ~(KVRING_FLAG_HOST_ONLY | KVRING_FLAG_NAIVE_UPKEEP | KVRING_FLAG_ROPE_3D))
        return fail(nullptr, KVRING_EINVAL, "unknown flag bits");
    if (c->flags & KVRING_FLAG_ROPE_3D) {
        if (c->frame_tokens < 1 || c->frame_width < 1 || c->frame_tokens % c->frame_width != 0)
            return fail(nullptr, KVRING_EINVAL, "3-D RoPE: frame_tokens and frame_width must be >= 1, frame_width dividing frame_tokens");
        if (c->capacity % c->frame_tokens != 0)
            return fail(nullptr, KVRING_EINVAL, "3-D RoPE: capacity must be a whole number of frames");
        const int half = c->head_dim / 2;
        if (c->rope_pairs_t != 0 || c->rope_pairs_h != 0) {
            if (c->rope_pairs_t < 1 || c->rope_pairs_h < 1 || c->rope_pairs_t + c->rope_pairs_h > half - 1)
                return fail(nullptr, KVRING_EINVAL, "3-D RoPE: each band needs at least one pair (pt + ph <= d/2 - 1)");
        }
    }
    return KVRING_OK;
}

int choose_splits(const kvring_t* r, int units, int ntiles) {
    int best = 1;
    long long best_cost = -1;
    const long long slots = (long long)r->num_sms;   // one attention CTA per SM
    for (int s = 1; s <= std::min(std::min(r->max_splits, 4), ntiles); ++s) {   // at most 4 (the merge's limit)
        const int tps = (ntiles + s - 1) / s;
        const int se = (ntiles + tps - 1) / tps;
        const long long waves = ((long long)units * se + slots - 1) / slots;
        const long long cost = waves * tps * 8 + (se > 1 ? 1 : 0);   // tile-times, plus a small charge for combining
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = se; }
    }
    return best;
}

// Write or rewrite on a naive-upkeep ring (arguments already checked): the window
// is shifted by a copy (write) or its newest rows replaced (rewrite); positions
// and chunk ids of the window rows are kept in logical order.
int naive_write(kvring_t* r, int layer, const void* k, const void* v, int n, bool rewrite, void* stream) {
    const kvring_config& c = r->cfg;
    LayerState& L = r->layers[layer];
    const int R = c.capacity;
    const int64_t drop = rewrite ? 0 : std::max<int64_t>(0, L.count + n - R);
    const int64_t keep = rewrite ? L.count - n : L.count - drop;
    if (!r->host_only) {
        const int H = c.num_heads, d = c.head_dim;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        WriteParams w{};
        w.k = static_cast<const uint16_t*>(k);
        w.v = static_cast<const uint16_t*>(v);
        w.T = n;
        w.H = H;
        w.d = d;
        w.amax_tokens_per_block = write_amax_tokens_per_block(H, d);
        w.amax_blocks = (n + w.amax_tokens_per_block - 1) / w.amax_tokens_per_block;
        w.part = r->wpart;
        cudaError_t e = launch_write_amax(w, s);
        if (e != cudaSuccess) return cuda_fail(r, e, "write amax kernel launch");
        const size_t win = (size_t)H * r->Rpad * d, am = (size_t)H * r->Rpad;
        const size_t per_buf = (size_t)c.num_layers;
        const int src = L.cur, dst = rewrite ? L.cur : 1 - L.cur;
        NaiveAppendParams p{};
        p.k = w.k;
        p.v = w.v;
        p.kw_src = r->kwin + (src * per_buf + layer) * win;
        p.vw_src = r->vwin + (src * per_buf + layer) * win;
        p.kw_dst = r->kwin + (dst * per_buf + layer) * win;
        p.vw_dst = r->vwin + (dst * per_buf + layer) * win;
        p.ka_src = r->kaw + (src * per_buf + layer) * am;
        p.va_src = r->vaw + (src * per_buf + layer) * am;
        p.ka_dst = r->kaw + (dst * per_buf + layer) * am;
        p.va_dst = r->vaw + (dst * per_buf + layer) * am;
        p.part = r->wpart;
        p.amax_blocks = w.amax_blocks;
        p.T = n;
        p.H = H;
        p.d = d;
        p.Rpad = (int)r->Rpad;
        p.keep = (int)keep;
        p.drop = (int)drop;
        p.row_begin = rewrite ? (int)keep : 0;
        e = launch_naive_append(p, s);
        if (e != cudaSuccess) return cuda_fail(r, e, "naive append kernel launch");
        r->launches += 2;
        L.cur = dst;
    }
    L.fresh = false;
    if (rewrite) return KVRING_OK;
    // window rows in logical order: the kept rows move up by `drop`, the chunk follows
    for (int64_t row = 0; row < keep; ++row) {
        L.pos[row] = L.pos[row + drop];
        L.chunk[row] = L.chunk[row + drop];
    }
    for (int j = 0; j < n; ++j) {
        L.pos[keep + j] = (int32_t)(L.next_pos + j);
        L.chunk[keep + j] = (int32_t)L.writes;
    }
    L.last_pos = L.next_pos;
    L.last_n = n;
    L.count = keep + n;
    L.head = L.count % R;
    L.next_pos += n;
    L.writes += 1;
    return KVRING_OK;
}

}  // namespace

namespace kvring_impl {
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return KVRING_ECUDA;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult res = encode(map, dtype, (cuuint32_t)rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? KVRING_OK : KVRING_ECUDA;
}

// Message reported by kvring_last_error(NULL) for calls that have no ring.
void set_thread_error(const std::string& msg) { g_create_error = msg; }

// 3-D tiled tensor map over uint8 data (the rings and Q tiles); KVRING_OK or KVRING_ECUDA.
int encode_u8_map(CUtensorMap* map, void* base, const cuuint64_t dims[3], const cuuint64_t strides[2],
                  const cuuint32_t box[3], CUtensorMapSwizzle swz) {
    return make_map(nullptr, map, base, dims, strides, box, swz);
}
}  // namespace kvring_impl

extern "C" {

int kvring_create(const kvring_config* cfg_in, kvring_t** out) {
    if (!out) return fail(nullptr, KVRING_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = check_config(cfg_in);
    if (rc) return rc;
    kvring_config cfg = *cfg_in;
    if (cfg.max_position == 0) cfg.max_position = 65536;
    if (cfg.rope_theta == 0.f) cfg.rope_theta = 10000.f;
    if (cfg.max_position < cfg.max_tokens_per_write)
        return fail(nullptr, KVRING_EINVAL, "max_position must be >= max_tokens_per_write");

    kvring_t* r = new (std::nothrow) kvring_t();
    if (!r) return fail(nullptr, KVRING_ENOMEM, "host allocation failed");
    r->cfg = cfg;
    r->host_only = (cfg.flags & KVRING_FLAG_HOST_ONLY) != 0;
    r->naive = (cfg.flags & KVRING_FLAG_NAIVE_UPKEEP) != 0;
    r->rope3d = (cfg.flags & KVRING_FLAG_ROPE_3D) != 0;
    if (r->rope3d && cfg.rope_pairs_t == 0 && cfg.rope_pairs_h == 0) {
        cfg.rope_pairs_h = cfg.head_dim / 6;
        cfg.rope_pairs_t = cfg.head_dim / 2 - 2 * cfg.rope_pairs_h;
        r->cfg = cfg;
    }
    r->Rpad = round_up(cfg.capacity, 128);
    r->Tstride = round_up(cfg.max_tokens_per_write, 256);
    r->layers.resize(cfg.num_layers);
    for (auto& l : r->layers) {
        l.pos.assign(cfg.capacity, -1);
        l.chunk.assign(cfg.capacity, -1);
    }
    if (r->host_only) { *out = r; return KVRING_OK; }

    cudaError_t e = cudaGetDevice(&r->device);
    cudaDeviceProp prop{};
    if (e == cudaSuccess) e = cudaGetDeviceProperties(&prop, r->device);
    if (e != cudaSuccess) { delete r; return fail(nullptr, KVRING_ENODEV, std::string("no CUDA device: ") + cudaGetErrorString(e)); }
    if (prop.major * 10 + prop.minor != 103) {
        delete r;
        return fail(nullptr, KVRING_ENODEV, "device is sm_" + std::to_string(prop.major * 10 + prop.minor) + ", this library is built for sm_103a");
    }
    r->num_sms = prop.multiProcessorCount;

    const int64_t L = cfg.num_layers, H = cfg.num_heads, d = cfg.head_dim;
    const int64_t ntiles_max = r->Rpad / 128, npairs_max = r->Tstride / 256;
    r->max_splits = (int)std::max<int64_t>(1, std::min<int64_t>(ntiles_max, (4 * r->num_sms + H * npairs_max - 1) / (H * npairs_max)));
    // asked here, once, so that no attention call makes the occupancy query
    for (int sp = 2; sp <= 4; ++sp) r->cluster_cap[sp] = attend_max_clusters((int)d, sp);
    const size_t ring_bytes = (size_t)(L * H * r->Rpad * d);
    const size_t amax_bytes = (size_t)(L * H * r->Rpad) * sizeof(float);
    const size_t rope_bytes = (size_t)cfg.max_position * (d / 2) * sizeof(float2);
    struct { void** p; size_t n; } allocs[] = {
        {(void**)&r->k8, ring_bytes}, {(void**)&r->vt8, ring_bytes},
        {(void**)&r->kamax, amax_bytes}, {(void**)&r->vamax, amax_bytes},
        {(void**)&r->rope, rope_bytes},
        {(void**)&r->q8, (size_t)(H * r->Tstride * d)}, {(void**)&r->qamax, (size_t)(H * r->Tstride) * sizeof(float)},
        {(void**)&r->part_o, (size_t)(r->max_splits * H * r->Tstride * d) * sizeof(float)},
        {(void**)&r->part_ml, (size_t)(r->max_splits * H * r->Tstride * 2) * sizeof(float)},
        {(void**)&r->counters, (size_t)(2 * H * npairs_max) * sizeof(int)},
        {(void**)&r->wpart, (size_t)(2 * H) * sizeof(float) *
                                (size_t)((cfg.max_tokens_per_write + write_amax_tokens_per_block((int)H, (int)d) - 1) /
                                         write_amax_tokens_per_block((int)H, (int)d))},
        {(void**)&r->err, 4 * sizeof(int)},
    };
    const size_t win_bytes = r->naive ? 2 * ring_bytes * sizeof(uint16_t) : 0;
    const size_t winam_bytes = r->naive ? 2 * amax_bytes : 0;
    struct { void** p; size_t n; } naive_allocs[] = {
        {(void**)&r->kwin, win_bytes}, {(void**)&r->vwin, win_bytes},
        {(void**)&r->kaw, winam_bytes}, {(void**)&r->vaw, winam_bytes},
    };
    for (auto& a : naive_allocs) {
        if (a.n == 0) continue;
        e = cudaMalloc(a.p, a.n);
        if (e != cudaSuccess) { free_device(r); delete r; return fail(nullptr, KVRING_ENOMEM, std::string("cudaMalloc: ") + cudaGetErrorString(e)); }
        e = cudaMemset(*a.p, 0, a.n);
        if (e != cudaSuccess) { free_device(r); delete r; return fail(nullptr, KVRING_ECUDA, std::string("cudaMemset: ") + cudaGetErrorString(e)); }
    }
    for (auto& a : allocs) {
        e = cudaMalloc(a.p, a.n);
        if (e != cudaSuccess) { free_device(r); delete r; return fail(nullptr, KVRING_ENOMEM, std::string("cudaMalloc: ") + cudaGetErrorString(e)); }
        e = cudaMemset(*a.p, 0, a.n);
        if (e != cudaSuccess) { free_device(r); delete r; return fail(nullptr, KVRING_ECUDA, std::string("cudaMemset: ") + cudaGetErrorString(e)); }
    }
    {
        std::vector<float2> tab;
        const Rope3D r3{cfg.frame_tokens, cfg.frame_width, cfg.rope_pairs_t, cfg.rope_pairs_h};
        build_rope_table(tab, cfg.max_position, (int)d, (double)cfg.rope_theta, r->rope3d ? &r3 : nullptr);
        e = cudaMemcpy(r->rope, tab.data(), rope_bytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) { free_device(r); delete r; return fail(nullptr, KVRING_ECUDA, std::string("cudaMemcpy: ") + cudaGetErrorString(e)); }
    }
    // TMA tensor maps over the rings and the Q scratch
    {
        const CUtensorMapSwizzle swz_d = d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        const cuuint64_t kdims[3] = {(cuuint64_t)d, (cuuint64_t)r->Rpad, (cuuint64_t)(L * H)};
        const cuuint64_t kstr[2] = {(cuuint64_t)d, (cuuint64_t)(r->Rpad * d)};
        const cuuint32_t kbox[3] = {(cuuint32_t)d, 128, 1};
        const cuuint64_t vdims[3] = {(cuuint64_t)r->Rpad, (cuuint64_t)d, (cuuint64_t)(L * H)};
        const cuuint64_t vstr[2] = {(cuuint64_t)r->Rpad, (cuuint64_t)(r->Rpad * d)};
        const cuuint32_t vbox[3] = {128, (cuuint32_t)d, 1};
        const cuuint64_t qdims[3] = {(cuuint64_t)d, (cuuint64_t)r->Tstride, (cuuint64_t)H};
        const cuuint64_t qstr[2] = {(cuuint64_t)d, (cuuint64_t)(r->Tstride * d)};
        const cuuint32_t qbox[3] = {(cuuint32_t)d, 128, 1};
        if ((rc = make_map(nullptr, &r->maps.k8, r->k8, kdims, kstr, kbox, swz_d)) ||
            (rc = make_map(nullptr, &r->maps.vt8, r->vt8, vdims, vstr, vbox, CU_TENSOR_MAP_SWIZZLE_128B)) ||
            (rc = make_map(nullptr, &r->maps.q8, r->q8, qdims, qstr, qbox, swz_d)) ||
            (cudaSuccess != write_setup() && (rc = fail(nullptr, KVRING_ECUDA, "write kernel attributes"))) ||
            ((rc = write_rope_map(&r->rope_map, r->rope, cfg.max_position, (int)d)) &&
             (rc = fail(nullptr, rc, "tensor map of the RoPE table")))) {
            free_device(r);
            delete r;
            return rc;
        }
    }
    *out = r;
    return KVRING_OK;
}

int kvring_destroy(kvring_t* r) {
    if (!r) return KVRING_OK;
    if (!r->host_only) free_device(r);
    delete r;
    return KVRING_OK;
}

int kvring_write_ex(kvring_t* r, int32_t layer, const void* k, const void* v, int32_t n,
                    uint32_t flags, void* stream) {
    if (!r) return KVRING_EINVAL;
    const kvring_config& c = r->cfg;
    if (layer < 0 || layer >= c.num_layers) return fail(r, KVRING_EINVAL, "layer out of range");
    if (flags & ~KVRING_WRITE_REWRITE) return fail(r, KVRING_EINVAL, "unknown write flag");
    if (n < 0 || n > c.max_tokens_per_write) return fail(r, KVRING_EINVAL, "n_tokens out of range [0, max_tokens_per_write]");
    if (r->rope3d && n % c.frame_tokens != 0)
        return fail(r, KVRING_EINVAL, "3-D RoPE: n_tokens must be a whole number of frames");
    LayerState& L = r->layers[layer];
    const bool rewrite = (flags & KVRING_WRITE_REWRITE) != 0;
    if (rewrite && L.writes == 0) return fail(r, KVRING_ESTATE, "rewrite before any write to this layer");
    if (rewrite && n != L.last_n) return fail(r, KVRING_ESTATE, "a rewrite must have the latest write's n_tokens");
    if (n == 0) return KVRING_OK;
    if (!r->host_only && (!k || !v)) return fail(r, KVRING_EINVAL, "k or v is NULL");
    if (!r->host_only && ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15))
        return fail(r, KVRING_EINVAL, "k and v must be 16-byte aligned");
    if (!rewrite && L.next_pos + n > c.max_position)
        return fail(r, KVRING_ESTATE, "positions would reach max_position: call kvring_rebase first");
    if (r->naive) return naive_write(r, layer, k, v, n, rewrite, stream);
    const int R = c.capacity;
    // first slot and position of the chunk written: the next ones, or the latest chunk's again
    const int64_t slot0 = rewrite ? (L.head - n + R) % R : L.head;
    const int64_t pos0 = rewrite ? L.last_pos : L.next_pos;
    if (!r->host_only) {
        WriteParams p{};
        p.k = static_cast<const uint16_t*>(k);
        p.v = static_cast<const uint16_t*>(v);
        const size_t lh = (size_t)layer * c.num_heads;
        p.k8 = r->k8 + lh * r->Rpad * c.head_dim;
        p.vt8 = r->vt8 + lh * r->Rpad * c.head_dim;
        p.kamax = r->kamax + lh * r->Rpad;
        p.vamax = r->vamax + lh * r->Rpad;
        p.rope = r->rope;
        p.head = slot0;
        p.pos0 = pos0;
        p.T = n;
        p.H = c.num_heads;
        p.d = c.head_dim;
        p.R = R;
        p.Rpad = (int)r->Rpad;
        p.ngroups_ring = (R + 15) / 16;
        p.group0 = (int)(slot0 / 16);
        // 16-slot groups touched by slots [slot0, slot0 + n) mod R
        const int64_t end = slot0 + n;
        int groups;
        if (end <= R) {
            groups = (int)((end - 1) / 16 - slot0 / 16 + 1);
        } else {
            const int64_t g1 = p.ngroups_ring - slot0 / 16;
            const int64_t g2 = (end - R - 1) / 16 + 1;
            groups = (int)std::min<int64_t>(p.ngroups_ring, g1 + g2);
        }
        p.groups = groups;
        p.amax_tokens_per_block = write_amax_tokens_per_block(p.H, p.d);
        p.amax_blocks = (n + p.amax_tokens_per_block - 1) / p.amax_tokens_per_block;
        p.part = r->wpart;
        p.err = r->err;
        p.timeout_ns = r->debug_write_timeout_ns > 0 ? r->debug_write_timeout_ns : 2000000000LL;
        p.skip_group = r->debug_skip_group;
        r->debug_skip_group = -1;
        r->debug_write_timeout_ns = 0;
        p.ropemap = r->rope_map;
        if (write_input_maps(p) != KVRING_OK) return fail(r, KVRING_ECUDA, "tensor maps of the chunk's K and V");
        cudaError_t e = launch_write(p, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(r, e, "write kernel launch");
        r->launches += 1;
    }
    if (rewrite) return KVRING_OK;   // same slots, positions and chunk id: nothing moves
    for (int j = 0; j < n; ++j) {
        const int64_t slot = (L.head + j) % R;
        L.pos[slot] = (int32_t)(L.next_pos + j);
        L.chunk[slot] = (int32_t)L.writes;
    }
    L.last_pos = L.next_pos;
    L.last_n = n;
    L.head = (L.head + n) % R;
    L.count = std::min<int64_t>(L.count + n, R);
    L.next_pos += n;
    L.writes += 1;
    return KVRING_OK;
}

int kvring_write(kvring_t* r, int32_t layer, const void* k, const void* v, int32_t n, void* stream) {
    return kvring_write_ex(r, layer, k, v, n, 0u, stream);
}

int kvring_attend(kvring_t* r, int32_t layer, const void* q, int32_t n_q, float* out, void* stream) {
    if (!r) return KVRING_EINVAL;
    const kvring_config& c = r->cfg;
    if (r->host_only) return fail(r, KVRING_EINVAL, "attend is not available on a host-only ring");
    if (layer < 0 || layer >= c.num_layers) return fail(r, KVRING_EINVAL, "layer out of range");
    if (n_q < 0 || n_q > c.max_tokens_per_write) return fail(r, KVRING_EINVAL, "n_q out of range");
    if (n_q == 0) return KVRING_OK;
    if (!q || !out) return fail(r, KVRING_EINVAL, "q or out is NULL");
    const LayerState& L = r->layers[layer];
    if (L.writes == 0 || L.count == 0) return fail(r, KVRING_ESTATE, "attend before any write to this layer");
    if (n_q != L.last_n) return fail(r, KVRING_ESTATE, "n_q must equal the latest write's n_tokens");
    if (r->naive && !L.fresh)
        return fail(r, KVRING_ESTATE, "naive-upkeep ring: kvring_naive_refresh is due after a write, rewrite or rebase");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int d = c.head_dim, H = c.num_heads;
    const int Tpad = (int)round_up(n_q, 128);

    QPrepParams qp{};
    qp.q = static_cast<const uint16_t*>(q);
    qp.q8 = r->q8;
    qp.qamax = r->qamax;
    qp.rope = r->rope;
    qp.pos0 = L.last_pos;
    qp.T = n_q;
    qp.Tpad = Tpad;
    qp.H = H;
    qp.d = d;
    qp.Tstride = (int)r->Tstride;
    cudaError_t e = launch_qprep(qp, s);
    if (e != cudaSuccess) return cuda_fail(r, e, "q-prep kernel launch");
    r->launches += 1;

    AttendParams ap{};
    const size_t lh = (size_t)layer * H;
    ap.kamax = r->kamax + lh * r->Rpad;
    ap.vamax = r->vamax + lh * r->Rpad;
    ap.qamax = r->qamax;
    ap.out = out;
    ap.part_o = r->part_o;
    ap.part_ml = r->part_ml;
    ap.counters = r->counters;
    ap.err = r->err;
    ap.T = n_q;
    ap.H = H;
    ap.d = d;
    ap.Rpad = (int)r->Rpad;
    ap.Tstride = (int)r->Tstride;
    ap.count = (int)L.count;
    ap.layer = layer;
    ap.npairs = (n_q + 255) / 256;
    ap.ntiles = (int)((L.count + 127) / 128);
    ap.splits = choose_splits(r, H * ap.npairs, ap.ntiles);
    ap.tiles_per_split = (ap.ntiles + ap.splits - 1) / ap.splits;
    ap.splits = (ap.ntiles + ap.tiles_per_split - 1) / ap.tiles_per_split;
    ap.log2e_rsqrt_d = (float)(1.4426950408889634 / std::sqrt((double)d));
    ap.timeout_ns = r->debug_timeout_ns > 0 ? r->debug_timeout_ns : 2000000000LL;
    ap.skip_tile = r->debug_skip_tile;
    // The splits of a (head, pair) merge through distributed shared memory when
    // they can run as one cluster and every cluster fits on the device at once;
    // else, with every CTA resident at once (one per SM), through global memory
    // together; else the last split to finish merges them.
    const int units = H * ap.npairs;
    ap.cluster = 0;
    if (ap.splits > 1 && ap.splits <= 4) ap.cluster = r->cluster_cap[ap.splits] >= units ? 1 : 0;
    ap.coop = (!ap.cluster && ap.splits > 1 && units * ap.splits <= r->num_sms) ? 1 : 0;
    r->debug_skip_tile = -1;
    r->debug_timeout_ns = 0;
    e = launch_attend(ap, r->maps, s);
    if (e != cudaSuccess) return cuda_fail(r, e, "attention kernel launch");
    r->launches += 1;
    r->last_q_rows = n_q;
    return KVRING_OK;
}

int kvring_rebase(kvring_t* r, void* stream) {
    if (!r) return KVRING_EINVAL;
    const kvring_config& c = r->cfg;
    RebaseParams p{};
    bool any = false;
    for (int l = 0; l < c.num_layers; ++l) {
        const LayerState& L = r->layers[l];
        const int64_t delta = L.next_pos - L.count;
        p.delta[l] = (int)delta;
        p.count[l] = (int)L.count;
        any = any || (delta != 0 && L.count > 0);
    }
    if (!r->host_only && any && !r->naive) {   // a naive ring rotates at every refresh instead
        p.k8 = r->k8;
        p.kamax = r->kamax;
        p.rope = r->rope;
        p.L = c.num_layers;
        p.H = c.num_heads;
        p.d = c.head_dim;
        p.Rpad = (int)r->Rpad;
        // 3-D: a reset moves whole frames and turns only the time pairs
        p.pairs = r->rope3d ? c.rope_pairs_t : c.head_dim / 2;
        cudaError_t e = launch_rebase(p, r->num_sms, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(r, e, "rebase kernel launch");
        r->launches += 1;
    }
    for (int l = 0; l < c.num_layers; ++l) {
        LayerState& L = r->layers[l];
        const int64_t delta = L.next_pos - L.count;
        if (delta != 0)
            for (auto& ps : L.pos)
                if (ps >= 0) ps -= (int32_t)delta;
        L.last_pos -= delta;
        L.next_pos = L.count;
        if (delta != 0) L.fresh = false;
    }
    r->resets += 1;
    return KVRING_OK;
}

int kvring_naive_refresh(kvring_t* r, int32_t layer, void* stream) {
    if (!r) return KVRING_EINVAL;
    const kvring_config& c = r->cfg;
    if (!r->naive) return fail(r, KVRING_EINVAL, "not a naive-upkeep ring (KVRING_FLAG_NAIVE_UPKEEP)");
    if (layer < 0 || layer >= c.num_layers) return fail(r, KVRING_EINVAL, "layer out of range");
    LayerState& L = r->layers[layer];
    if (L.writes == 0 || L.count == 0) return fail(r, KVRING_ESTATE, "refresh before any write to this layer");
    if (!r->host_only) {
        const int H = c.num_heads, d = c.head_dim;
        const size_t win = (size_t)H * r->Rpad * d, am = (size_t)H * r->Rpad;
        const size_t buf = (size_t)L.cur * c.num_layers + layer;
        NaiveRefreshParams p{};
        p.kw = r->kwin + buf * win;
        p.vw = r->vwin + buf * win;
        p.ka = r->kaw + buf * am;
        p.va = r->vaw + buf * am;
        p.k8 = r->k8 + (size_t)layer * win;
        p.vt8 = r->vt8 + (size_t)layer * win;
        p.kamax = r->kamax + (size_t)layer * am;
        p.vamax = r->vamax + (size_t)layer * am;
        p.rope = r->rope;
        p.pos0 = L.next_pos - L.count;
        p.count = (int)L.count;
        p.H = H;
        p.d = d;
        p.Rpad = (int)r->Rpad;
        cudaError_t e = launch_naive_refresh(p, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(r, e, "naive refresh kernel launch");
        r->launches += 1;
    }
    L.fresh = true;
    return KVRING_OK;
}

int kvring_get_state(const kvring_t* r, int32_t layer, kvring_state* out) {
    if (!r || !out) return KVRING_EINVAL;
    if (layer < 0 || layer >= r->cfg.num_layers) return fail(const_cast<kvring_t*>(r), KVRING_EINVAL, "layer out of range");
    const LayerState& L = r->layers[layer];
    out->head = L.head;
    out->count = L.count;
    out->next_pos = L.next_pos;
    out->writes = L.writes;
    out->resets = r->resets;
    out->last_write_pos = L.last_pos;
    out->last_write_tokens = L.last_n;
    return KVRING_OK;
}

int kvring_snapshot(const kvring_t* rc, int32_t layer, uint8_t* hk, uint8_t* hv, float* hka, float* hva,
                    int32_t* hpos, int32_t* hchunk, void* stream) {
    kvring_t* r = const_cast<kvring_t*>(rc);
    if (!r) return KVRING_EINVAL;
    const kvring_config& c = r->cfg;
    if (layer < 0 || layer >= c.num_layers) return fail(r, KVRING_EINVAL, "layer out of range");
    const LayerState& L = r->layers[layer];
    if (hpos) std::memcpy(hpos, L.pos.data(), sizeof(int32_t) * c.capacity);
    if (hchunk) std::memcpy(hchunk, L.chunk.data(), sizeof(int32_t) * c.capacity);
    if (!hk && !hv && !hka && !hva) return KVRING_OK;
    if (r->host_only) return fail(r, KVRING_EINVAL, "no device data on a host-only ring");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t H = c.num_heads, d = c.head_dim, R = c.capacity, Rp = r->Rpad;
    const size_t lh = (size_t)layer * H;
    cudaError_t e = cudaSuccess;
    std::vector<uint8_t> vt;
    if (hk) e = cudaMemcpy2DAsync(hk, R * d, r->k8 + lh * Rp * d, Rp * d, R * d, H, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && hv) {
        vt.resize(H * d * R);
        e = cudaMemcpy2DAsync(vt.data(), R, r->vt8 + lh * Rp * d, Rp, R, H * d, cudaMemcpyDeviceToHost, s);
    }
    if (e == cudaSuccess && hka)
        e = cudaMemcpy2DAsync(hka, R * sizeof(float), r->kamax + lh * Rp, Rp * sizeof(float), R * sizeof(float), H, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && hva)
        e = cudaMemcpy2DAsync(hva, R * sizeof(float), r->vamax + lh * Rp, Rp * sizeof(float), R * sizeof(float), H, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(r, e, "snapshot copy");
    if (hv)
        for (size_t h = 0; h < H; ++h)
            for (size_t dd = 0; dd < d; ++dd)
                for (size_t sl = 0; sl < R; ++sl) hv[(h * R + sl) * d + dd] = vt[(h * d + dd) * R + sl];
    return KVRING_OK;
}

int kvring_snapshot_q(const kvring_t* rc, uint8_t* hq, float* hqamax, void* stream) {
    kvring_t* r = const_cast<kvring_t*>(rc);
    if (!r) return KVRING_EINVAL;
    if (r->host_only) return fail(r, KVRING_EINVAL, "no device data on a host-only ring");
    if (r->last_q_rows <= 0) return fail(r, KVRING_ESTATE, "no attention call yet");
    if (!hq && !hqamax) return KVRING_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t H = r->cfg.num_heads, d = r->cfg.head_dim, n = (size_t)r->last_q_rows, ts = (size_t)r->Tstride;
    cudaError_t e = cudaSuccess;
    if (hq) e = cudaMemcpy2DAsync(hq, n * d, r->q8, ts * d, n * d, H, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && hqamax)
        e = cudaMemcpy2DAsync(hqamax, n * sizeof(float), r->qamax, ts * sizeof(float), n * sizeof(float), H,
                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(r, e, "Q snapshot copy");
    return KVRING_OK;
}

int kvring_check_device(kvring_t* r, void* stream) {
    if (!r) return KVRING_EINVAL;
    if (r->host_only) return KVRING_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int w[4] = {0, 0, 0, 0};
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(w, r->err, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(r, e, "reading the device error word");
    if (w[0] == 0) return KVRING_OK;
    static const char* sites[] = {"?", "Q tiles", "K/V stage full", "K/V stage free", "S", "P", "O", "fp16 V full",
                                  "fp16 V free", "the other KV splits"};
    static const char* write_sites[] = {"?", "the chunk's rows", "the chunk amax from the cluster"};
    if (w[1] == kKernelWrite) {
        const int site = (w[2] >= 0 && w[2] <= 2) ? w[2] : 0;
        r->error = std::string("device wait timed out in the write kernel (wait for ") + write_sites[site] +
                   ", block " + std::to_string(w[3]) + ")";
    } else {
        const int site = (w[2] >= 0 && w[2] <= 9) ? w[2] : 0;
        r->error = std::string("device wait timed out in the attention kernel (wait for ") + sites[site] +
                   ", block " + std::to_string(w[3]) + ")";
    }
    e = cudaMemset(r->err, 0, sizeof(w));
    // a CTA that gave up may have left a split counter behind
    if (e == cudaSuccess)
        e = cudaMemset(r->counters, 0, 2 * (size_t)r->cfg.num_heads * (r->Tstride / 256) * sizeof(int));
    if (e != cudaSuccess) return cuda_fail(r, e, "clearing the device error word");
    return KVRING_ETIMEOUT;
}

const char* kvring_last_error(const kvring_t* r) {
    if (!r) return g_create_error.c_str();
    return r->error.c_str();
}

int kvring_launch_count(const kvring_t* r, uint64_t* out) {
    if (!r || !out) return KVRING_EINVAL;
    *out = r->launches;
    return KVRING_OK;
}

int kvring_debug_fault(kvring_t* r, int32_t skip_tile, int64_t timeout_ns) {
    if (!r) return KVRING_EINVAL;
    if (skip_tile < -1 || timeout_ns < 0) return fail(r, KVRING_EINVAL, "skip_tile >= -1 and timeout_ns >= 0 required");
    r->debug_skip_tile = skip_tile;
    r->debug_timeout_ns = timeout_ns;
    return KVRING_OK;
}

int kvring_debug_fault_write(kvring_t* r, int32_t skip_group, int64_t timeout_ns) {
    if (!r) return KVRING_EINVAL;
    if (skip_group < -1 || timeout_ns < 0) return fail(r, KVRING_EINVAL, "skip_group >= -1 and timeout_ns >= 0 required");
    r->debug_skip_group = skip_group;
    r->debug_write_timeout_ns = timeout_ns;
    return KVRING_OK;
}

}  // extern "C"
