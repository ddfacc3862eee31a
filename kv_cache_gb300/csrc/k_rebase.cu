// K2: position-reset rebase -- one delta rotation of every cached K, in place.
//
// The pages reset positions every 42 steps and, at each reset, apply a single
// delta rotation to the cached window instead of recomputing it (ai.info,
// "Characters funziona in tempo reale su quattro H100", section "La gestione della
// cache spostata al momento della scrittura"; neurocartel.com, "Runway Characters
// realtime on 4 H100", section "Кэш: 240 attention calls и работа на запись").
//
// Each code is de-quantised with its slot's frozen scale, the pair is rotated by
// -delta (cos(delta*w_i), -sin(delta*w_i), read from the RoPE table row `delta`)
// and re-quantised with the same scale.  V has no RoPE and is not touched.
// One launch covers every layer: a block takes one (layer, head, 128-slot block)
// unit at a time; units of layers with delta == 0 and slots past the layer's
// count are skipped.  16-byte loads and stores, HBM-bound.
#include "common.cuh"
#include "kvring_internal.h"

namespace kvring_impl {


// Each thread handles kItems 16-byte pieces of a unit, all in the same column
// chunk (the block's thread count is a multiple of the chunks per row), and
// issues every load (the codes, their slots' amax, the chunk's rotation entries
// -- one RoPE table row per layer, read through L1) before it uses any, so a
// unit costs one memory round trip; no shared memory and no barriers.
constexpr int kItems = 8;
constexpr int kRebaseThreadsR = 128;   // threads per block; 128 * kItems = 1024 pieces = one 128-slot unit at d = 128

// kPartial: some pairs of a row do not turn (3-D RoPE); their bytes are kept.
template <bool kPartial>
__global__ void __launch_bounds__(kRebaseThreadsR) rebase_kernel(const __grid_constant__ RebaseParams p) {
    const int d = p.d;
    const int c16n = d / 16;
    const int nsb = p.Rpad / 128;
    const long long units = (long long)p.L * p.H * nsb;
    const int tid = threadIdx.x;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const int lh = (int)(u / nsb);
        const int sb = (int)(u - (long long)lh * nsb);
        const int l = lh / p.H;
        const int delta = p.delta[l];
        const int cnt = p.count[l];
        if (delta == 0 || sb * 128 >= cnt) continue;     // uniform over the block
        const int nslots = min(128, cnt - sb * 128);
        uint8_t* base = p.k8 + ((size_t)lh * p.Rpad + (size_t)sb * 128) * d;
        const float* am = p.kamax + (size_t)lh * p.Rpad + (size_t)sb * 128;
        const float4* rot = reinterpret_cast<const float4*>(p.rope + (size_t)delta * (d / 2));   // (cos, sin) pairs
        const int c = tid % c16n;   // this thread's column chunk, the same for all its pieces
        if (kPartial && c * 8 >= p.pairs) continue;   // no pair of this chunk turns (past the time band)
        float4 cs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) cs[e] = __ldg(rot + c * 4 + e);   // pairs 8c + 2e, 8c + 2e + 1
        uint4 w[kItems];
        float amax[kItems];
        bool live[kItems];
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            const int r = (tid + k * kRebaseThreadsR) / c16n;
            live[k] = r < nslots;
            if (live[k]) {
                w[k] = *reinterpret_cast<const uint4*>(base + (size_t)r * d + c * 16);
                amax[k] = __ldg(am + r);
            }
        }
#pragma unroll
        for (int k = 0; k < kItems; ++k) {
            if (!live[k]) continue;
            const int r = (tid + k * kRebaseThreadsR) / c16n;
            const float sc = scale_of(amax[k]), iv = inv_of(amax[k]);
            const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f0 = e4m3x2_to_float2(ws[e] & 0xFFFFu);
                const float2 f1 = e4m3x2_to_float2(ws[e] >> 16);
                float y0, y1, z0, z1;
                // rotation by -delta: cos unchanged, sine negated
                rope_pair(__fmul_rn(f0.x, sc), __fmul_rn(f0.y, sc), cs[e].x, -cs[e].y, y0, y1);
                rope_pair(__fmul_rn(f1.x, sc), __fmul_rn(f1.y, sc), cs[e].z, -cs[e].w, z0, z1);
                out[e] = e4m3x2(__fmul_rn(y0, iv), __fmul_rn(y1, iv)) |
                         (e4m3x2(__fmul_rn(z0, iv), __fmul_rn(z1, iv)) << 16);
                // pairs past the ones that turn keep their bytes (3-D RoPE: the
                // height and width bands of the chunk holding the band edge)
                if (kPartial) {
                    const int pair0 = c * 8 + 2 * e;
                    if (pair0 >= p.pairs) out[e] = ws[e];
                    else if (pair0 + 1 >= p.pairs) out[e] = (out[e] & 0xFFFFu) | (ws[e] & 0xFFFF0000u);
                }
            }
            *reinterpret_cast<uint4*>(base + (size_t)r * d + c * 16) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

// 3-D RoPE with the time band in the first four 16-byte pieces of a row (pt <= 32
// pairs): only those pieces move.  Every thread takes one piece column
// c = tid % 4 of 8 rows, so a block covers 256 rows (two 128-slot blocks) of one
// (layer, head) and keeps as many bytes in flight as a block of the full-row
// kernel; pairs past the time band in the last piece keep their bytes.
constexpr int kTbCols = 4, kTbItems = 8, kTbRows = kRebaseThreadsR / kTbCols * kTbItems;   // 256

__global__ void __launch_bounds__(kRebaseThreadsR) rebase_time_band_kernel(const __grid_constant__ RebaseParams p) {
    const int d = p.d;
    const int nrb = (p.Rpad + kTbRows - 1) / kTbRows;
    const int lh = (int)(blockIdx.x / nrb);
    const int rb = (int)(blockIdx.x - (unsigned)lh * nrb);
    const int l = lh / p.H;
    const int delta = p.delta[l];
    const int cnt = p.count[l];
    const int c = threadIdx.x % kTbCols;
    if (delta == 0 || rb * kTbRows >= cnt || c * 8 >= p.pairs) return;
    uint8_t* base = p.k8 + (size_t)lh * p.Rpad * d;
    const float* am = p.kamax + (size_t)lh * p.Rpad;
    const float4* rot = reinterpret_cast<const float4*>(p.rope + (size_t)delta * (d / 2));
    float4 cs[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) cs[e] = __ldg(rot + c * 4 + e);
    uint4 w[kTbItems];
    float amax[kTbItems];
#pragma unroll
    for (int k = 0; k < kTbItems; ++k) {
        const int r = rb * kTbRows + (int)threadIdx.x / kTbCols + k * (kRebaseThreadsR / kTbCols);
        if (r < cnt) {
            w[k] = *reinterpret_cast<const uint4*>(base + (size_t)r * d + c * 16);
            amax[k] = __ldg(am + r);
        }
    }
#pragma unroll
    for (int k = 0; k < kTbItems; ++k) {
        const int r = rb * kTbRows + (int)threadIdx.x / kTbCols + k * (kRebaseThreadsR / kTbCols);
        if (r >= cnt) continue;
        const float sc = scale_of(amax[k]), iv = inv_of(amax[k]);
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
        uint32_t out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int pair0 = c * 8 + 2 * e;
            const float2 f0 = e4m3x2_to_float2(ws[e] & 0xFFFFu);
            const float2 f1 = e4m3x2_to_float2(ws[e] >> 16);
            float y0, y1, z0, z1;
            rope_pair(__fmul_rn(f0.x, sc), __fmul_rn(f0.y, sc), cs[e].x, -cs[e].y, y0, y1);
            rope_pair(__fmul_rn(f1.x, sc), __fmul_rn(f1.y, sc), cs[e].z, -cs[e].w, z0, z1);
            out[e] = e4m3x2(__fmul_rn(y0, iv), __fmul_rn(y1, iv)) |
                     (e4m3x2(__fmul_rn(z0, iv), __fmul_rn(z1, iv)) << 16);
            if (pair0 >= p.pairs) out[e] = ws[e];
            else if (pair0 + 1 >= p.pairs) out[e] = (out[e] & 0xFFFFu) | (ws[e] & 0xFFFF0000u);
        }
        *reinterpret_cast<uint4*>(base + (size_t)r * d + c * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

cudaError_t launch_rebase(const RebaseParams& p, int num_sms, cudaStream_t s) {
    if (p.pairs < p.d / 2 && p.pairs <= 8 * kTbCols) {
        const long long units = (long long)p.L * p.H * ((p.Rpad + kTbRows - 1) / kTbRows);
        rebase_time_band_kernel<<<(unsigned)units, kRebaseThreadsR, 0, s>>>(p);
        return cudaGetLastError();
    }
    // one unit per block: the blocks in flight then cover one contiguous stretch of
    // the rings (measured faster than a persistent or grid-stride layout)
    (void)num_sms;
    const long long units = (long long)p.L * p.H * (p.Rpad / 128);
    long long grid = units;
    if (grid > 0x7fffffffLL) grid = 0x7fffffffLL;
    if (grid < 1) grid = 1;
    if (p.pairs < p.d / 2)
        rebase_kernel<true><<<(unsigned)grid, kRebaseThreadsR, 0, s>>>(p);
    else
        rebase_kernel<false><<<(unsigned)grid, kRebaseThreadsR, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvring_impl
