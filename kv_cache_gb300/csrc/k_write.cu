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
// Two launches, chained on the stream by programmatic dependent launch:
//   write_amax_kernel   reads the chunk's K and V once, from HBM; block b stores
//                       its per-head maximum of K (pair norms) and of V (|v|) as
//                       partial [K|V][b][H].  Plain stores, no atomics.
//   write_store_kernel  one block per (16-slot ring group, head, K|V): fetches
//                       its rows (still in L2) and, for K, their RoPE rows while
//                       the first kernel runs; after the grid dependency it
//                       reduces its head's partials to the chunk amax, rotates K,
//                       quantises and stores -- K rows as 16-byte pieces of
//                       [H][Rpad][d], V as one 16-byte run of 16 slots per (head,
//                       column) of the slot-contiguous [H][d][Rpad] ring.  Slots
//                       of a partly covered group that belong to older chunks are
//                       left alone.
// The first kernel lets the second start only after its own grid dependency has
// resolved, so by then the inputs are final and the second may read them before
// its own wait; the partials it reads only after that wait.  No thread waits on
// another thread of its grid.
#include "common.cuh"
#include "kvring_internal.h"

namespace kvring_impl {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxLoads = 4;          // 16-byte loads in flight per thread
constexpr int kStoreThreads = 128;

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

// ---------------------------------------------------------------- quantise + store
// d <= 128: a K group is 16 rows x d/16 pieces <= 128 items, one per thread; a V
// group is 16 rows x d/8 pieces, staged in shared memory.
__global__ void __launch_bounds__(kStoreThreads) write_store_kernel(const __grid_constant__ WriteParams p) {
    __shared__ __align__(16) uint16_t sv[16 * 128];     // V: the group's 16 rows of this head
    __shared__ int s_tok[16];
    __shared__ float s_red[kStoreThreads / 32];
    const int h = blockIdx.y;
    const bool is_v = blockIdx.z == 1;
    const int tid = threadIdx.x;
    const int d = p.d, H = p.H;
    int g = p.group0 + (int)blockIdx.x;
    if (g >= p.ngroups_ring) g -= p.ngroups_ring;
    if (tid < 16) s_tok[tid] = group_token(p, g, tid);
    __syncthreads();
    const size_t in_row = (size_t)H * d;           // elements per token
    // This grid starts only after every block of the amax grid is past its grid
    // dependency, so the chunk's K and V are final: fetch them now.
    const int c16n = d / 16;
    const int j = tid / c16n, c = tid - j * c16n;  // K item of this thread (j < 16 when valid)
    const int t = tid < 16 * c16n ? s_tok[j] : -1;
    uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
    float4 cs[4];
    if (!is_v) {
        if (t >= 0) {
            const uint4* x = reinterpret_cast<const uint4*>(p.k + (size_t)t * in_row + (size_t)h * d + c * 16);
            const float4* tab = reinterpret_cast<const float4*>(p.rope + (size_t)(p.pos0 + t) * (d / 2) + c * 8);
            a = __ldg(x);
            b = __ldg(x + 1);
#pragma unroll
            for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + e);   // pairs 2e and 2e + 1 of the piece
        }
    } else {
        const int per_row = d / 8;
        for (int it = tid; it < 16 * per_row; it += kStoreThreads) {
            const int jj = it / per_row, cc = it - jj * per_row;
            const int tt = s_tok[jj];
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (tt >= 0) w = __ldg(reinterpret_cast<const uint4*>(p.v + (size_t)tt * in_row + (size_t)h * d) + cc);
            *reinterpret_cast<uint4*>(sv + jj * d + cc * 8) = w;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // chunk amax of (K|V, h): the maximum of the amax grid's partials
    const float* part = p.part + (size_t)(is_v ? p.amax_blocks : 0) * H + h;
    float m = 0.f;
    for (int i = tid; i < p.amax_blocks; i += kStoreThreads) m = fmaxf(m, part[(size_t)i * H]);
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) s_red[tid >> 5] = m;
    __syncthreads();
    float amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kStoreThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
    const float inv = inv_of(amax);
    if (!is_v) {
        if (t >= 0) {
            const uint32_t ws[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float y0, y1, z0, z1;
                rope_pair(bf16_lo(ws[2 * e]), bf16_hi(ws[2 * e]), cs[e].x, cs[e].y, y0, y1);
                rope_pair(bf16_lo(ws[2 * e + 1]), bf16_hi(ws[2 * e + 1]), cs[e].z, cs[e].w, z0, z1);
                out[e] = e4m3x2(__fmul_rn(y0, inv), __fmul_rn(y1, inv)) |
                         (e4m3x2(__fmul_rn(z0, inv), __fmul_rn(z1, inv)) << 16);
            }
            *reinterpret_cast<uint4*>(p.k8 + ((size_t)h * p.Rpad + g * 16 + j) * d + c * 16) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
        if (tid < 16 && s_tok[tid] >= 0) p.kamax[(size_t)h * p.Rpad + g * 16 + tid] = amax;
        return;
    }
    // V: one 16-slot run per column
    uint32_t owned = 0;                             // bit j: slot j of the group belongs to this chunk
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) owned |= (s_tok[jj] >= 0 ? 1u : 0u) << jj;
    for (int dd = tid; dd < d; dd += kStoreThreads) {
        uint32_t words[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float v0 = bf16_lo(sv[(4 * q + 0) * d + dd]), v1 = bf16_lo(sv[(4 * q + 1) * d + dd]);
            const float v2 = bf16_lo(sv[(4 * q + 2) * d + dd]), v3 = bf16_lo(sv[(4 * q + 3) * d + dd]);
            words[q] = e4m3x2(__fmul_rn(v0, inv), __fmul_rn(v1, inv)) |
                       (e4m3x2(__fmul_rn(v2, inv), __fmul_rn(v3, inv)) << 16);
        }
        uint8_t* dst = p.vt8 + ((size_t)h * d + dd) * p.Rpad + g * 16;
        if (owned == 0xFFFFu) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        } else {
            for (int jj = 0; jj < 16; ++jj)
                if (owned & (1u << jj)) dst[jj] = (uint8_t)(words[jj / 4] >> (8 * (jj % 4)));
        }
    }
    if (tid < 16 && s_tok[tid] >= 0) p.vamax[(size_t)h * p.Rpad + g * 16 + tid] = amax;
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

cudaError_t launch_write(const WriteParams& p, cudaStream_t s) {
    cudaError_t e = launch_write_amax(p, s);
    if (e != cudaSuccess) return e;
    const dim3 g2((unsigned)p.groups, (unsigned)p.H, 2);
    return launch_pdl(reinterpret_cast<const void*>(write_store_kernel), g2, dim3(kStoreThreads), 0, s, p);
}

}  // namespace kvring_impl
