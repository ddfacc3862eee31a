// K1: write one chunk into a layer's ring -- RoPE on K, per-(head, chunk) amax,
// FP8 e4m3 quantisation, store into the ring slots.
//
// The pages move RoPE and FP8 quantisation to the moment a chunk enters the cache
// and keep the cache as a ring buffer, so nothing is copied as the window advances
// (ai.info, "Characters funziona in tempo reale su quattro H100", section "La
// gestione della cache spostata al momento della scrittura"; neurocartel.com,
// "Runway Characters realtime on 4 H100", section "Кэш: 240 attention calls и
// работа на запись").
//
// One launch, one thread-block cluster of kWriteCluster CTAs per (head, K|V):
//   each CTA takes a share of the chunk's 16-slot ring groups, loads its rows of
//   that head once with TMA (one 16-row box per group; K also the RoPE rows of
//   those positions) into shared memory and takes their maximum (K: RoPE-pair
//   norms, V: |v|); it pushes that partial into every CTA of the cluster with
//   remote stores that complete on the receiver's mbarrier, and once its own
//   barrier holds all of them it quantises and stores from shared memory -- K
//   rows as 4-byte pieces of [H][Rpad][d], V as one 16-byte run of 16 slots per
//   (head, column) of the slot-contiguous [H][d][Rpad] ring.  Slots of a partly
//   covered group that belong to older chunks are left alone.  No CTA reads
//   another's shared memory, and each leaves only after every value meant for
//   it has arrived.
// write_amax_kernel, the chunk amax alone (partials per block in global memory),
// serves the naive-upkeep comparison scheme.
#include "common.cuh"
#include "kvring_internal.h"
#include "tc.cuh"

namespace kvring_impl {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxLoads = 4;          // 16-byte loads in flight per thread
constexpr int kWriteCluster = 8;            // CTAs per (head, K|V)
constexpr int kWriteThreads = 256;
// rows of a CTA: a chunk of at most 2048 tokens touches at most 130 ring groups
constexpr int kWriteMaxGroupsPerCta = (2048 / 16 + 2 + kWriteCluster - 1) / kWriteCluster;
constexpr int kWriteMaxRows = kWriteMaxGroupsPerCta * 16;
constexpr int kWritePdl = 0;                // programmatic dependent launch: off (back-to-back writes measured slower with it)
constexpr int kWritePrefetch = 14;          // K items per thread kept in registers (757 tokens need 14)

// ---------------------------------------------------------------- amax pass
// Block b covers tokens [b * tpb, (b + 1) * tpb) of K (blockIdx.y == 0) or V: a
// contiguous run of the token-major [T][H][d] input.  One head row is d/8
// consecutive 16-byte pieces, so the lanes of a warp fall into aligned groups of
// d/8 lanes that share a head; the group reduces by shuffles and its first lane
// folds the result into a shared per-head maximum.
__global__ void __launch_bounds__(kAmaxThreads) write_amax_kernel(const __grid_constant__ WriteParams p) {
    extern __shared__ uint32_t s_head_max[];   // [H], float bits (amax >= 0 orders like its bits)
    const bool is_v = blockIdx.y == 1;
    const int tid = threadIdx.x;
    const int H = p.H, d = p.d;
    const int per_row = d / 8;                 // 16-byte pieces per head row: 8 or 16
    const int per_token = H * per_row;
    const int first = (int)blockIdx.x * p.amax_tokens_per_block * per_token;
    const int last = min(first + p.amax_tokens_per_block * per_token, p.T * per_token);
    for (int h = tid; h < H; h += kAmaxThreads) s_head_max[h] = 0u;
    // the previous grid in the stream may still run: read nothing before it ends;
    // the next grid may start once every block is past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? p.v : p.k);
    for (int base = first; base < last; base += kAmaxThreads * kAmaxLoads) {
        uint4 w[kAmaxLoads];
#pragma unroll
        for (int k = 0; k < kAmaxLoads; ++k) {
            const int q = base + tid + k * kAmaxThreads;
            w[k] = q < last ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kAmaxLoads; ++k) {
            const int q = base + tid + k * kAmaxThreads;
            const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
            float m = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = bf16_lo(ws[e]), x1 = bf16_hi(ws[e]);
                m = is_v ? fmaxf(m, fmaxf(fabsf(x0), fabsf(x1))) : fmaxf(m, pair_norm(x0, x1));
            }
            // reduce over the d/8 lanes of this head row (whole warp: all lanes take part)
            for (int off = per_row >> 1; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if ((tid & (per_row - 1)) == 0 && q < last) atomicMax(&s_head_max[(q / per_row) % H], __float_as_uint(m));
        }
    }
    __syncthreads();
    float* part = p.part + ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * H;
    for (int h = tid; h < H; h += kAmaxThreads) part[h] = __uint_as_float(s_head_max[h]);
}

// Token written to slot j of ring group g by this chunk, or -1.
__device__ __forceinline__ int group_token(const WriteParams& p, int g, int j) {
    const int s = g * 16 + j;
    if (s >= p.R) return -1;
    int t = s - (int)p.head;
    if (t < 0) t += p.R;
    return t < p.T ? t : -1;
}

// ---------------------------------------------------------------- one-launch write
enum : int { kWaitWriteRows = 1, kWaitWriteAmax = 2 };

// Ring group of the CTA's local group index gi.
__device__ __forceinline__ int local_group(const WriteParams& p, int gb, int gi) {
    const int g = p.group0 + gb + gi;
    return g >= p.ngroups_ring ? g - p.ngroups_ring : g;
}

// max of two bf16 pairs, lane by lane; a NaN lane yields the other operand's lane
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ void write_timed_out(const WriteParams& p, int site) {
    if (atomicCAS(p.err, 0, KVRING_ETIMEOUT) == 0) {
        p.err[1] = kKernelWrite;
        p.err[2] = site;
        p.err[3] = (int)blockIdx.x;
    }
}

// Pairs 2q and 2q + 1 of a K row (x, bf16) rotated by their RoPE entries (cs).
__device__ __forceinline__ float4 rotate2(uint2 x, float4 cs) {
    float4 y;
    rope_pair(bf16_lo(x.x), bf16_hi(x.x), cs.x, cs.y, y.x, y.y);
    rope_pair(bf16_lo(x.y), bf16_hi(x.y), cs.z, cs.w, y.z, y.w);
    return y;
}
__device__ __forceinline__ uint32_t quant4(float4 y, float inv) {
    return e4m3x2(__fmul_rn(y.x, inv), __fmul_rn(y.y, inv)) | (e4m3x2(__fmul_rn(y.z, inv), __fmul_rn(y.w, inv)) << 16);
}

// Ring slot of row r of a CTA whose first group is gb.
__device__ __forceinline__ int row_slot(const WriteParams& p, int gb, int r) {
    return local_group(p, gb, r / 16) * 16 + (r % 16);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
                 : "memory");
}

// The ring's grid: one cluster of kWriteCluster CTAs per (head, K|V); CTA `rank`
// of a cluster takes ring groups [groups * rank / C, groups * (rank + 1) / C) of
// the chunk, rows_max = 16 * ceil(groups / C) rows at most.
//
// Loading: one TMA box of 16 rows per group, from the tensor map of the chunk
// ({d, H, T}, box {d, 1, 16}) at the token of the group's first slot counted
// without wrapping (t0 = 16 g - head, + R when the whole group lies before
// head).  A slot of an older chunk then falls outside [0, T) and reads zeros,
// and the slots past R of the ring's last group read a duplicate of a row that
// some other slot takes: neither changes the maximum.  The one exception, a
// chunk of more than R - 16 tokens whose end wraps into the group of its first
// slot, is patched with plain loads.  K also takes, per group, the 16 RoPE rows
// of those positions (nothing writes the table after the ring is created, so
// they are fetched before the grid dependency).
//
// Each CTA takes the maximum of its rows (K: the squared RoPE-pair norm -- its
// square root, which keeps the order, is taken once at the end; V: |v|),
// pushes it into every CTA of the cluster with remote stores that count on the
// receiver's mbarrier, and quantises once its own barrier has all of them.
//   K  rotates its first kWritePrefetch 2-pair items per thread while the
//      maxima travel, then quantises them and stores 4 bytes each of [H][Rpad][d];
//   V  stores one 16-slot run per (group, column), 16 bytes of [H][d][Rpad].
// Shared memory: srow [rows_max][D] bf16, then K's stab [rows_max][D / 2] float2.
template <int D>
__global__ void __launch_bounds__(kWriteThreads) write_cluster_kernel(const __grid_constant__ WriteParams p) {
    extern __shared__ __align__(128) uint8_t wsm[];
    __shared__ __align__(8) uint64_t bars[2];          // [0] the rows have landed, [1] the cluster's maxima
    __shared__ float sred[kWriteThreads / 32];
    __shared__ uint32_t spart[kWriteCluster];          // every CTA's maximum (float bits)
    __shared__ uint32_t sowned[kWriteMaxGroupsPerCta]; // bit j set when slot j of the group is this chunk's
    constexpr int Q = D / 4;                           // K items (2 pairs, 8 bytes) of a row
    const int tid = threadIdx.x, lane = tid & 31;
    const int rank = (int)(blockIdx.x % kWriteCluster);   // a cluster's CTAs are consecutive blocks
    const int cid = (int)(blockIdx.x / kWriteCluster);
    const bool is_v = (cid & 1) != 0;
    const int h = cid >> 1;
    const int gb = (int)((long long)p.groups * rank / kWriteCluster);
    const int ng = (int)((long long)p.groups * (rank + 1) / kWriteCluster) - gb;
    const int rows = ng * 16;
    const int rows_max = (p.groups + kWriteCluster - 1) / kWriteCluster * 16;
    uint16_t* srow = reinterpret_cast<uint16_t*>(wsm);
    float2* stab = reinterpret_cast<float2*>(srow + (size_t)rows_max * D);
    if (tid == kWriteThreads - 32) {   // the last warp: warp 0 issues the loads
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_expect_tx(&bars[0], (uint32_t)(rows * D * (is_v ? 2 : 6)));   // the arrival and every box's bytes
        mbar_expect_tx(&bars[1], kWriteCluster * 4);                       // the arrival; the bytes come from the cluster
        fence_mbar_init();
    }
    // first half of a cluster barrier; its second half, before the exchange,
    // makes sure every CTA of the cluster has started and set up its barriers
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // which slots of each group are this chunk's: one ballot per 32 rows
    for (int r0 = tid & ~31; r0 < rows; r0 += kWriteThreads) {
        const int r = r0 + lane;
        const bool mine = r < rows && group_token(p, local_group(p, gb, r / 16), r % 16) >= 0;
        const uint32_t b = __ballot_sync(0xffffffffu, mine);
        if (lane == 0) {
            sowned[r0 / 16] = b & 0xFFFFu;
            if (r0 + 16 < rows) sowned[r0 / 16 + 1] = b >> 16;
        }
    }
    __syncthreads();   // the barriers are set up
    // lane gi of warp 0 loads group gi
    int t0 = 0;
    if (tid < ng) {
        const int g = local_group(p, gb, tid);
        t0 = g * 16 - (int)p.head + (g * 16 + 15 < p.head ? p.R : 0);
        if (!is_v) tma_load_2d(stab + (size_t)tid * 16 * (D / 2), &p.ropemap, &bars[0], 0, (int)(p.pos0 + t0));
    }
    // the chunk's K and V may come from the grid before: wait for it; the next
    // grid may start now (it waits for this one the same way)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid < ng && local_group(p, gb, tid) != p.skip_group)
        tma_load_3d(srow + (size_t)tid * 16 * D, is_v ? &p.vmap : &p.kmap, &bars[0], 0, h, t0);
    bool ok = mbar_wait(&bars[0], 0, p.timeout_ns);
    if (!ok) write_timed_out(p, kWaitWriteRows);
    if (__syncthreads_and(ok) == 0) ok = false;
    // a chunk of more than R - 16 tokens: slots before head in head's group hold its last tokens
    const int hg = (int)(p.head / 16), hj = (int)(p.head % 16);
    if (ok && p.T > p.R - 16 && hj != 0) {
        const int gi = (hg - p.group0 - gb + p.ngroups_ring) % p.ngroups_ring;
        if (gi < ng) {
            for (int e = tid; e < hj * (D / 8); e += kWriteThreads) {
                const int j = e / (D / 8), c = e % (D / 8);
                const int t = hg * 16 + j - (int)p.head + p.R;
                if (t >= p.T) continue;
                const uint4* src = reinterpret_cast<const uint4*>((is_v ? p.v : p.k) + ((size_t)t * p.H + h) * D);
                reinterpret_cast<uint4*>(srow + (size_t)(gi * 16 + j) * D)[c] = src[c];
                if (!is_v) {   // 16 bytes of row data take 32 bytes of RoPE entries
                    const uint4* tab = reinterpret_cast<const uint4*>(p.rope + (size_t)(p.pos0 + t) * (D / 2));
                    uint4* dst = reinterpret_cast<uint4*>(stab + (size_t)(gi * 16 + j) * (D / 2));
                    dst[2 * c] = tab[2 * c];
                    dst[2 * c + 1] = tab[2 * c + 1];
                }
            }
        }
        __syncthreads();
    }
    // this CTA's maximum
    float m = 0.f;
    if (ok) {
        const uint4* rows16 = reinterpret_cast<const uint4*>(srow);
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        uint32_t m2 = 0u;
        for (int base = tid; base < rows * (D / 8); base += 4 * kWriteThreads) {
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int idx = base + u * kWriteThreads;
                w[u] = idx < rows * (D / 8) ? rows16[idx] : zero;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (is_v) {
                    m2 = bf16x2_max(m2, bf16x2_max(w[u].x & 0x7FFF7FFFu, w[u].y & 0x7FFF7FFFu));
                    m2 = bf16x2_max(m2, bf16x2_max(w[u].z & 0x7FFF7FFFu, w[u].w & 0x7FFF7FFFu));
                } else {
                    const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x0 = bf16_lo(ws[e]), x1 = bf16_hi(ws[e]);
                        m = fmaxf(m, __fadd_rn(__fmul_rn(x0, x0), __fmul_rn(x1, x1)));
                    }
                }
            }
        }
        if (is_v) m = fmaxf(bf16_lo(m2), bf16_hi(m2));
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) sred[tid >> 5] = m;
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (tid < kWriteCluster) {
        float cm = sred[0];
#pragma unroll
        for (int w = 1; w < kWriteThreads / 32; ++w) cm = fmaxf(cm, sred[w]);
        const uint32_t dst = dsmem_map(smem_u32(spart + rank), (uint32_t)tid);
        const uint32_t rbar = dsmem_map(smem_u32(&bars[1]), (uint32_t)tid);
        asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                     ::"r"(dst), "r"(__float_as_uint(cm)), "r"(rbar) : "memory");
    }
    // K: rotate while the maxima travel
    float4 y[kWritePrefetch];
    if (!is_v && ok) {
#pragma unroll
        for (int k = 0; k < kWritePrefetch; ++k) {
            const int idx = tid + k * kWriteThreads;
            const bool in = idx < rows * Q;
            const uint2 xx = in ? *reinterpret_cast<const uint2*>(srow + (size_t)idx * 4) : make_uint2(0u, 0u);
            const float4 cs = in ? *reinterpret_cast<const float4*>(stab + (size_t)idx * 2) : make_float4(0.f, 0.f, 0.f, 0.f);
            y[k] = rotate2(xx, cs);
        }
    }
    // each CTA exits only after all eight maxima have reached it, so no remote
    // store arrives later.  A CTA whose rows timed out pushes its value only after
    // that wait (at most timeout_ns), so this wait is given twice that and 1 ms
    // more: every value pushed arrives before any CTA gives up here.
    const bool got = mbar_wait(&bars[1], 0, 2 * p.timeout_ns + 1000000LL);
    if (!got) write_timed_out(p, kWaitWriteAmax);
    if (__syncthreads_and(got && ok) == 0) {
        if (!ok) mbar_wait(&bars[0], 0, p.timeout_ns);   // no box left in flight into this CTA (bounded again)
        return;
    }
    float amax = __uint_as_float(spart[0]);
#pragma unroll
    for (int r = 1; r < kWriteCluster; ++r) amax = fmaxf(amax, __uint_as_float(spart[r]));
    if (!is_v) amax = __fsqrt_rn(amax);
    const float inv = inv_of(amax);
    if (!is_v) {
        uint8_t* k8 = p.k8 + (size_t)h * p.Rpad * D;
        uint32_t code[kWritePrefetch];
#pragma unroll
        for (int k = 0; k < kWritePrefetch; ++k) code[k] = quant4(y[k], inv);
#pragma unroll
        for (int k = 0; k < kWritePrefetch; ++k) {
            const int idx = tid + k * kWriteThreads;
            const int r = idx / Q;
            const bool mine = idx < rows * Q && ((sowned[min(r, rows_max - 1) / 16] >> (r % 16)) & 1u);
            if (mine) *reinterpret_cast<uint32_t*>(k8 + (size_t)row_slot(p, gb, r) * D + (idx % Q) * 4) = code[k];
        }
        for (int idx = tid + kWritePrefetch * kWriteThreads; idx < rows * Q; idx += kWriteThreads) {
            const int r = idx / Q;
            if ((sowned[r / 16] >> (r % 16)) & 1u) {
                const float4 yy = rotate2(*reinterpret_cast<const uint2*>(srow + (size_t)idx * 4),
                                          *reinterpret_cast<const float4*>(stab + (size_t)idx * 2));
                *reinterpret_cast<uint32_t*>(k8 + (size_t)row_slot(p, gb, r) * D + (idx % Q) * 4) = quant4(yy, inv);
            }
        }
    } else {
        // V: columns 2c and 2c + 1 of a group, one 16-slot run each
        constexpr int C = D / 2;
        for (int idx = tid; idx < ng * C; idx += kWriteThreads) {
            const int gi = idx / C, c = idx % C;
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = *reinterpret_cast<const uint32_t*>(srow + (size_t)(gi * 16 + 4 * q + e) * D + 2 * c);
                lo[q] = e4m3x2(__fmul_rn(bf16_lo(w[0]), inv), __fmul_rn(bf16_lo(w[1]), inv)) |
                        (e4m3x2(__fmul_rn(bf16_lo(w[2]), inv), __fmul_rn(bf16_lo(w[3]), inv)) << 16);
                hi[q] = e4m3x2(__fmul_rn(bf16_hi(w[0]), inv), __fmul_rn(bf16_hi(w[1]), inv)) |
                        (e4m3x2(__fmul_rn(bf16_hi(w[2]), inv), __fmul_rn(bf16_hi(w[3]), inv)) << 16);
            }
            const uint32_t owned = sowned[gi];
            uint8_t* dst = p.vt8 + ((size_t)h * D + 2 * c) * p.Rpad + local_group(p, gb, gi) * 16;
            if (owned == 0xFFFFu) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4*>(dst + p.Rpad) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            } else {
                for (int j = 0; j < 16; ++j)
                    if (owned & (1u << j)) {
                        dst[j] = (uint8_t)(lo[j / 4] >> (8 * (j % 4)));
                        dst[p.Rpad + j] = (uint8_t)(hi[j / 4] >> (8 * (j % 4)));
                    }
            }
        }
    }
    // the chunk amax of each of this CTA's slots
    float* amax_out = (is_v ? p.vamax : p.kamax) + (size_t)h * p.Rpad;
    for (int r = tid; r < rows; r += kWriteThreads)
        if ((sowned[r / 16] >> (r % 16)) & 1u) amax_out[row_slot(p, gb, r)] = amax;
}

static cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              const WriteParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<WriteParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int write_amax_tokens_per_block(int H, int d) {
    const int pieces = kAmaxThreads * kAmaxLoads;      // one round of loads per block
    const int per_token = H * d / 8;
    return per_token >= pieces ? 1 : pieces / per_token;
}

cudaError_t launch_write_amax(const WriteParams& p, cudaStream_t s) {
    const dim3 g1((unsigned)p.amax_blocks, 2);
    return launch_pdl(reinterpret_cast<const void*>(write_amax_kernel), g1, dim3(kAmaxThreads),
                      (size_t)p.H * sizeof(uint32_t), s, p);
}

// At most kWriteMaxRows rows: 204 KB at d = 128.
size_t write_cluster_smem(const WriteParams& p) {
    const size_t rows_max = (size_t)(p.groups + kWriteCluster - 1) / kWriteCluster * 16;
    return rows_max * (size_t)p.d * 6;
}

int write_input_maps(WriteParams& p) {
    const cuuint64_t dims[3] = {(cuuint64_t)p.d, (cuuint64_t)p.H, (cuuint64_t)p.T};
    const cuuint64_t str[2] = {(cuuint64_t)p.d * 2, (cuuint64_t)p.H * p.d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)p.d, 1, 16};
    int rc = encode_tiled(&p.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(p.k), dims, str, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc == KVRING_OK)
        rc = encode_tiled(&p.vmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(p.v), dims, str, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    return rc;
}

int write_rope_map(CUtensorMap* map, const float2* rope, int64_t max_position, int d) {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)max_position};
    const cuuint64_t str[1] = {(cuuint64_t)d * 4};
    const cuuint32_t box[2] = {(cuuint32_t)d, 16};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<float2*>(rope), dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t write_setup() {
    const void* fns[2] = {reinterpret_cast<const void*>(write_cluster_kernel<64>),
                          reinterpret_cast<const void*>(write_cluster_kernel<128>)};
    const int smem[2] = {kWriteMaxRows * 64 * 6, kWriteMaxRows * 128 * 6};
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = cudaSuccess;
        if (kWriteCluster > 8) e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_write_d(const WriteParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(kWriteCluster * 2 * p.H), 1, 1);
    cfg.blockDim = dim3(kWriteThreads, 1, 1);
    cfg.dynamicSmemBytes = write_cluster_smem(p);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = kWritePdl;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kWriteCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, write_cluster_kernel<D>, p);
}

// write_setup() must have run on the device (kvring_create does it).
cudaError_t launch_write(const WriteParams& p, cudaStream_t s) {
    if ((p.groups + kWriteCluster - 1) / kWriteCluster * 16 > kWriteMaxRows) return cudaErrorInvalidValue;
    return p.d == 128 ? launch_write_d<128>(p, s) : launch_write_d<64>(p, s);
}

}  // namespace kvring_impl
