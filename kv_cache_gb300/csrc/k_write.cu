// K1: write one chunk into a layer's ring -- RoPE on K, per-(head, chunk) amax,
// FP8 e4m3 quantisation, store into the ring slots.  One pass over the input.
//
// The pages move RoPE and FP8 quantisation to the moment a chunk enters the cache
// and keep the cache as a ring buffer, so nothing is copied as the window advances
// (ai.info, "Characters funziona in tempo reale su quattro H100", section "La
// gestione della cache spostata al momento della scrittura"; neurocartel.com,
// "Runway Characters realtime on 4 H100", section "Кэш: 240 attention calls и
// работа на запись").
//
// Launch: grid (CL, H, 2), one thread-block cluster of CL <= 16 CTAs per (head,
// K|V).  The chunk's slots are cut into 16-slot groups aligned in the ring
// (the V ring is slot-contiguous, so a group is one 16-byte store per head_dim
// row); the groups are dealt to the cluster's CTAs in ring order.  Each CTA
// pulls its rows (and, for K, their RoPE table rows) into shared memory with
// bulk TMA copies issued by the 32 lanes of warp 0, takes its local amax, the
// cluster reduces the amax through distributed shared memory, and each CTA
// quantises its rows from shared memory.  Input bytes are read once.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kvring_internal.h"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace kvring_impl {

constexpr int kWriteThreads = 256;

// Token written to the j-th slot of visit-order group k of this chunk, or -1.
__device__ __forceinline__ int group_slot_token(const WriteParams& p, int k, int j, int& slot) {
    int g = p.group0 + k;
    if (g >= p.ngroups_ring) g -= p.ngroups_ring;
    const int s = g * 16 + j;
    slot = s;
    if (s >= p.R) return -1;
    int t = s - (int)p.head;
    if (t < 0) t += p.R;
    return t < p.T ? t : -1;
}

__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kWriteThreads) write_kernel(const __grid_constant__ WriteParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float s_red[kWriteThreads / 32];
    __shared__ float s_amax;
    __shared__ __align__(8) uint64_t s_bar;

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int h = blockIdx.y;
    const bool is_v = blockIdx.z == 1;
    const int d = p.d;
    const int tid = threadIdx.x;
    const int k0 = rank * p.groups / CL;
    const int k1 = (rank + 1) * p.groups / CL;
    const int nloc = (k1 - k0) * 16;
    uint16_t* sx = reinterpret_cast<uint16_t*>(smem);                              // [nloc][d] bf16
    float2* stab = reinterpret_cast<float2*>(smem + (size_t)nloc * d * 2);          // [nloc][d/2] (K only)

    // ---- 1. bulk copies of this CTA's rows (and, for K, their RoPE table rows) into shared memory
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&s_bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // This grid may start before the one ahead of it in the stream has finished
    // (programmatic launch): the set-up above overlaps that grid's tail, and
    // nothing is read or written before it has finished.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    const uint16_t* src = is_v ? p.v : p.k;
    if (tid < 32) {
        uint32_t bytes = 0;
        for (int li = tid; li < nloc; li += 32) {
            int slot;
            if (group_slot_token(p, k0 + li / 16, li % 16, slot) >= 0) bytes += is_v ? 2 * d : 6 * d;
        }
        if (bytes) mbar_expect_tx_only(&s_bar, bytes);
        __syncwarp();
        for (int li = tid; li < nloc; li += 32) {
            int slot;
            const int t = group_slot_token(p, k0 + li / 16, li % 16, slot);
            if (t < 0) continue;
            bulk_g2s(sx + (size_t)li * d, src + ((size_t)t * p.H + h) * d, 2 * d, &s_bar);
            if (!is_v) bulk_g2s(stab + (size_t)li * (d / 2), p.rope + (size_t)(p.pos0 + t) * (d / 2), 4 * d, &s_bar);
        }
        __syncwarp();
        if (tid == 0) mbar_arrive1(&s_bar);
    }
    // bounded wait for the copies (2 s), then once more before giving up on them
    {
        uint32_t done = 0;
        for (int round = 0; round < 2 && !done; ++round) {
            const uint64_t t0 = globaltimer_ns();
            while (true) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                    : "=r"(done) : "r"(smem_u32(&s_bar)) : "memory");
                if (done || globaltimer_ns() - t0 > 2000000000ull) break;
            }
            if (!done && tid == 0 && atomicCAS(p.err, 0, KVRING_ETIMEOUT) == 0) {
                p.err[1] = kKernelWrite;
                p.err[2] = 1;
                p.err[3] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
            }
        }
    }

    // ---- 2. local amax (K: largest pair norm of the un-rotated pairs; V: largest |v|)
    const int vec_per_row = d / 8;
    float local = 0.f;
    for (int qq = tid; qq < nloc * vec_per_row; qq += kWriteThreads) {
        const int li = qq / vec_per_row, c = qq - li * vec_per_row;
        int slot;
        if (group_slot_token(p, k0 + li / 16, li % 16, slot) < 0) continue;
        const uint4 w = *reinterpret_cast<const uint4*>(sx + (size_t)li * d + c * 8);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = bf16_lo(ws[e]), x1 = bf16_hi(ws[e]);
            local = is_v ? fmaxf(local, fmaxf(fabsf(x0), fabsf(x1))) : fmaxf(local, pair_norm(x0, x1));
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) local = fmaxf(local, __shfl_xor_sync(0xffffffffu, local, off));
    if ((tid & 31) == 0) s_red[tid >> 5] = local;
    __syncthreads();
    if (tid == 0) {
        float m = 0.f;
        for (int w = 0; w < kWriteThreads / 32; ++w) m = fmaxf(m, s_red[w]);
        s_amax = m;
    }
    // ---- 3. chunk amax over the cluster (distributed shared memory)
    cluster.sync();
    float amax = 0.f;
    for (int r = 0; r < CL; ++r) amax = fmaxf(amax, *cluster.map_shared_rank(&s_amax, r));
    const float inv = inv_of(amax);

    // ---- 4. quantise and store
    if (!is_v) {
        const int c16n = d / 16;
        for (int qq = tid; qq < nloc * c16n; qq += kWriteThreads) {
            const int li = qq / c16n, c = qq - li * c16n;
            int slot;
            if (group_slot_token(p, k0 + li / 16, li % 16, slot) < 0) continue;
            const uint4* xs = reinterpret_cast<const uint4*>(sx + (size_t)li * d + c * 16);
            const uint4 a = xs[0], b = xs[1];
            const uint32_t ws[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            const float4* tab = reinterpret_cast<const float4*>(stab + (size_t)li * (d / 2) + c * 8);
            uint32_t out[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float4 cs = tab[e2];          // pairs 2*e2 and 2*e2+1
                float y0, y1, z0, z1;
                rope_pair(bf16_lo(ws[2 * e2]), bf16_hi(ws[2 * e2]), cs.x, cs.y, y0, y1);
                rope_pair(bf16_lo(ws[2 * e2 + 1]), bf16_hi(ws[2 * e2 + 1]), cs.z, cs.w, z0, z1);
                out[e2] = e4m3x2(__fmul_rn(y0, inv), __fmul_rn(y1, inv)) |
                          (e4m3x2(__fmul_rn(z0, inv), __fmul_rn(z1, inv)) << 16);
            }
            *reinterpret_cast<uint4*>(p.k8 + ((size_t)h * p.Rpad + slot) * d + c * 16) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
    } else {
        const int ng = k1 - k0;
        for (int qq = tid; qq < d * ng; qq += kWriteThreads) {
            const int kk = qq / d, dd = qq - kk * d;
            uint32_t words[4] = {0u, 0u, 0u, 0u};
            uint32_t written = 0;    // bit j: slot j of the group belongs to this chunk
            int slot0 = 0;
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                int s0, s1;
                const int t0 = group_slot_token(p, k0 + kk, j, s0);
                const int t1 = group_slot_token(p, k0 + kk, j + 1, s1);
                if (j == 0) slot0 = s0;
                const float v0 = t0 >= 0 ? bf16_lo(sx[(size_t)(kk * 16 + j) * d + dd]) : 0.f;
                const float v1 = t1 >= 0 ? bf16_lo(sx[(size_t)(kk * 16 + j + 1) * d + dd]) : 0.f;
                const uint32_t two = e4m3x2(__fmul_rn(v0, inv), __fmul_rn(v1, inv));
                words[j / 4] |= two << (8 * (j % 4));
                written |= (t0 >= 0 ? 1u : 0u) << j;
                written |= (t1 >= 0 ? 1u : 0u) << (j + 1);
            }
            uint8_t* dst = p.vt8 + ((size_t)h * d + dd) * p.Rpad + slot0;
            if (written == 0xFFFFu) {
                *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
            } else {
                for (int j = 0; j < 16; ++j)
                    if (written & (1u << j)) dst[j] = (uint8_t)(words[j / 4] >> (8 * (j % 4)));
            }
        }
    }
    float* am = is_v ? p.vamax : p.kamax;
    for (int li = tid; li < nloc; li += kWriteThreads) {
        int slot;
        const int t = group_slot_token(p, k0 + li / 16, li % 16, slot);
        if (t >= 0) am[(size_t)h * p.Rpad + slot] = amax;
    }
    // peers may still be reading s_amax
    cluster.sync();
}

cudaError_t launch_write(const WriteParams& p, cudaStream_t s) {
    // 16 CTAs per cluster (non-portable size, supported on this part) keep each
    // CTA's share small: ~4 groups (64 rows) for a 757-token chunk.
    const int CL = p.groups < 16 ? p.groups : 16;
    const int per = (p.groups + CL - 1) / CL;
    const size_t smem = (size_t)per * 16 * (size_t)p.d * 6;   // bf16 rows (2d bytes) + RoPE table rows (4d bytes)
    cudaError_t e = cudaFuncSetAttribute(write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(write_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, p.H, 2);
    cfg.blockDim = dim3(kWriteThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, write_kernel, p);
}

}  // namespace kvring_impl
