// The naive cache upkeep, kept as a measured comparison for the write-time ring.
//
// Before the change the pages describe, the serving code re-applied rotary
// embeddings to the whole cached window, re-quantised it and shifted it as the
// window advanced, on every attention call; moving that work to write time and
// keeping the cache as a ring took cache upkeep from 69.7 ms to 6.2 ms of a step
// (ai.info, "Characters funziona in tempo reale su quattro H100", section "La
// gestione della cache spostata al momento della scrittura"; wechild.cn news item,
// paragraph 7).  Two kernels:
//
//   naive_append_kernel   the shift: the window after a write is the kept rows
//                         of the old window (a copy, oldest dropped) followed by
//                         the new chunk; a rewrite replaces only the newest rows.
//                         Each row carries its chunk amax.
//   naive_refresh_kernel  the per-call upkeep: every row of the window is rotated
//                         at its current position, quantised with its chunk scale
//                         and stored in the layer's FP8 cache (row r -> slot r) in
//                         the layout the attention kernel reads.
//
// One block per (16 window rows, head); 16-byte loads and stores.
#include "common.cuh"
#include "kvring_internal.h"

namespace kvring_impl {

constexpr int kNaiveThreads = 128;

// ---------------------------------------------------------------- shift / append
// Launched after write_amax_kernel (programmatic dependent launch): that grid lets
// this one start only after its own grid dependency, so the inputs and the old
// window are final and the copies run at once; only the new rows' amax, which
// needs the first grid's partials, waits for it.
__global__ void __launch_bounds__(kNaiveThreads) naive_append_kernel(const __grid_constant__ NaiveAppendParams p) {
    __shared__ float s_red[2][kNaiveThreads / 32];
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int d = p.d, H = p.H;
    const int per_row = d / 8;                       // 16-byte pieces per row
    const int rows_end = p.keep + p.T;
    const int r0 = p.row_begin + (int)blockIdx.x * 16;
    const size_t in_row = (size_t)H * d;
    for (int it = tid; it < 16 * per_row; it += kNaiveThreads) {
        const int j = it / per_row, c = it - j * per_row;
        const int r = r0 + j;
        if (r >= rows_end) continue;
        uint4 wk, wv;
        if (r < p.keep) {
            const size_t src = ((size_t)h * p.Rpad + r + p.drop) * d + c * 8;
            wk = *reinterpret_cast<const uint4*>(p.kw_src + src);
            wv = *reinterpret_cast<const uint4*>(p.vw_src + src);
        } else {
            const size_t src = (size_t)(r - p.keep) * in_row + (size_t)h * d + c * 8;
            wk = __ldg(reinterpret_cast<const uint4*>(p.k + src));
            wv = __ldg(reinterpret_cast<const uint4*>(p.v + src));
        }
        const size_t dst = ((size_t)h * p.Rpad + r) * d + c * 8;
        *reinterpret_cast<uint4*>(p.kw_dst + dst) = wk;
        *reinterpret_cast<uint4*>(p.vw_dst + dst) = wv;
    }
    if (tid < 16) {
        const int r = r0 + tid;
        if (r < p.keep) {
            p.ka_dst[(size_t)h * p.Rpad + r] = p.ka_src[(size_t)h * p.Rpad + r + p.drop];
            p.va_dst[(size_t)h * p.Rpad + r] = p.va_src[(size_t)h * p.Rpad + r + p.drop];
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (r0 + 15 < p.keep) return;                    // no new rows in this block (uniform)
    // chunk amax of K and V for head h: the maximum of the first grid's partials
    float mk = 0.f, mv = 0.f;
    for (int i = tid; i < p.amax_blocks; i += kNaiveThreads) {
        mk = fmaxf(mk, p.part[(size_t)i * H + h]);
        mv = fmaxf(mv, p.part[(size_t)(p.amax_blocks + i) * H + h]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    }
    if ((tid & 31) == 0) {
        s_red[0][tid >> 5] = mk;
        s_red[1][tid >> 5] = mv;
    }
    __syncthreads();
    if (tid < 16) {
        const int r = r0 + tid;
        if (r >= p.keep && r < rows_end) {
            float ak = s_red[0][0], av = s_red[1][0];
#pragma unroll
            for (int w = 1; w < kNaiveThreads / 32; ++w) {
                ak = fmaxf(ak, s_red[0][w]);
                av = fmaxf(av, s_red[1][w]);
            }
            p.ka_dst[(size_t)h * p.Rpad + r] = ak;
            p.va_dst[(size_t)h * p.Rpad + r] = av;
        }
    }
}

// ---------------------------------------------------------------- per-call re-rotation + re-quantisation
// d <= 128: the K work of a block is 16 rows x d/16 pieces <= 128 items, one per
// thread; V rows are staged in shared memory and written as 16-slot runs.
__global__ void __launch_bounds__(kNaiveThreads) naive_refresh_kernel(const __grid_constant__ NaiveRefreshParams p) {
    __shared__ __align__(16) uint16_t sv[16 * 128];
    __shared__ float s_vinv[16];
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int d = p.d;
    const int r0 = (int)blockIdx.x * 16;
    // the window may have been written by the grid just before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int c16n = d / 16;
    const int j = tid / c16n, c = tid - j * c16n;
    const int r = r0 + j;
    if (tid < 16 * c16n && r < p.count) {
        const uint4* x = reinterpret_cast<const uint4*>(p.kw + ((size_t)h * p.Rpad + r) * d + c * 16);
        const float4* tab = reinterpret_cast<const float4*>(p.rope + (size_t)(p.pos0 + r) * (d / 2) + c * 8);
        const uint4 a = x[0], b = x[1];
        float4 cs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + e);   // pairs 2e and 2e + 1 of the piece
        const float amax = p.ka[(size_t)h * p.Rpad + r];
        const float inv = inv_of(amax);
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
        *reinterpret_cast<uint4*>(p.k8 + ((size_t)h * p.Rpad + r) * d + c * 16) =
            make_uint4(out[0], out[1], out[2], out[3]);
        if (c == 0) p.kamax[(size_t)h * p.Rpad + r] = amax;
    }
    // V: stage the 16 rows, then one 16-slot run per column
    const int per_row = d / 8;
    for (int it = tid; it < 16 * per_row; it += kNaiveThreads) {
        const int jj = it / per_row, cc = it - jj * per_row;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + jj < p.count) w = *reinterpret_cast<const uint4*>(p.vw + ((size_t)h * p.Rpad + r0 + jj) * d + cc * 8);
        *reinterpret_cast<uint4*>(sv + jj * d + cc * 8) = w;
    }
    if (tid < 16) {
        const int rr = r0 + tid;
        const float amax = rr < p.count ? p.va[(size_t)h * p.Rpad + rr] : 0.f;
        s_vinv[tid] = inv_of(amax);
        if (rr < p.count) p.vamax[(size_t)h * p.Rpad + rr] = amax;
    }
    __syncthreads();
    const int nrows = min(16, p.count - r0);
    for (int dd = tid; dd < d; dd += kNaiveThreads) {
        uint32_t words[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j0 = 4 * q;
            const float v0 = __fmul_rn(bf16_lo(sv[(j0 + 0) * d + dd]), s_vinv[j0 + 0]);
            const float v1 = __fmul_rn(bf16_lo(sv[(j0 + 1) * d + dd]), s_vinv[j0 + 1]);
            const float v2 = __fmul_rn(bf16_lo(sv[(j0 + 2) * d + dd]), s_vinv[j0 + 2]);
            const float v3 = __fmul_rn(bf16_lo(sv[(j0 + 3) * d + dd]), s_vinv[j0 + 3]);
            words[q] = e4m3x2(v0, v1) | (e4m3x2(v2, v3) << 16);
        }
        uint8_t* dst = p.vt8 + ((size_t)h * d + dd) * p.Rpad + r0;
        if (nrows == 16) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        } else {
            for (int jj = 0; jj < nrows; ++jj) dst[jj] = (uint8_t)(words[jj / 4] >> (8 * (jj % 4)));
        }
    }
}

static cudaError_t launch_pdl_naive(const void* fn, dim3 grid, void* arg, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kNaiveThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {arg};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_naive_append(const NaiveAppendParams& p, cudaStream_t s) {
    const int rows = p.keep + p.T - p.row_begin;
    const dim3 grid((unsigned)((rows + 15) / 16), (unsigned)p.H);
    return launch_pdl_naive(reinterpret_cast<const void*>(naive_append_kernel), grid,
                            const_cast<NaiveAppendParams*>(&p), s);
}

cudaError_t launch_naive_refresh(const NaiveRefreshParams& p, cudaStream_t s) {
    const dim3 grid((unsigned)((p.count + 15) / 16), (unsigned)p.H);
    return launch_pdl_naive(reinterpret_cast<const void*>(naive_refresh_kernel), grid,
                            const_cast<NaiveRefreshParams*>(&p), s);
}

}  // namespace kvring_impl
