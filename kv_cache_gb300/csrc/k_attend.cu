// K3 (Q prep), K4 (FP8 attention over the ring) and K5 (split combine).
//
// The pages have every attention call read a cache of 5,788 slots of which 757
// are new, 240 calls per step (wechild.cn news item on Runway's real-time
// Characters inference paper, paragraph 6; ai.info, "Characters funziona in
// tempo reale su quattro H100", section "La gestione della cache spostata al
// momento della scrittura"), and name the missing piece on Blackwell: an FP8
// attention kernel that accepts per-head scales (same article, section "Latenza
// dei turni e altre configurazioni GPU").
//
// K4 is one CTA of 128 threads per (head, 128-row query tile, KV split):
//  * Q (e4m3, from K3), K tiles [128 slots][d] and V tiles [d][128 slots] (e4m3)
//    arrive by TMA into 128-byte-swizzled shared memory, two K/V stages deep.
//  * S = Q K^T runs on tcgen05 (kind::f8f6f4, M = N = 128) into tensor memory.
//  * Thread i owns query row i (tensor-memory lane i): it reads S, applies the
//    per-slot K scale, keeps a running max m and sum l (online softmax; the max
//    is only moved when it grows by more than 2^8, so O is rarely rescaled),
//    and writes P = 2^(x - m) * (V scale of the slot / V scale reference) as
//    fp16 into shared memory.
//  * The V tile is widened from e4m3 to fp16 in shared memory (exact), and
//    O += P V runs on tcgen05 (kind::f16, M = 128, N = d) into tensor memory.
//  * Slots are walked in physical order 0..count-1: softmax attention does not
//    depend on key order and each slot already carries its rotation, so the
//    ring wrap needs no special case and no gather.
//  * Every wait is bounded; on a time-out the CTA records KVRING_ETIMEOUT in
//    the error word, drains its own copies and MMAs (bounded), frees its
//    tensor memory and returns.
#include "common.cuh"
#include "kvring_internal.h"
#include "tc.cuh"

namespace kvring_impl {

// ============================================================== K3: Q prep
// Rotate Q at the latest chunk's positions, quantise each (token, head) row to
// e4m3 with its own amax, write [H][Tstride][d] codes + [H][Tstride] amax.
// Rows T..Tpad-1 are written as zeros.
__global__ void __launch_bounds__(128) qprep_kernel(const __grid_constant__ QPrepParams p) {
    const int d = p.d;
    const int tpr = d / 8;                       // threads per row, 8 elements each
    const int rows_per_block = 128 / tpr;
    const int lrow = threadIdx.x / tpr;
    const int c = threadIdx.x % tpr;
    const int row = blockIdx.x * rows_per_block + lrow;   // over H * Tpad
    const bool in_range = row < p.H * p.Tpad;
    const int h = in_range ? row / p.Tpad : 0;
    const int t = in_range ? row % p.Tpad : 0;
    const bool real = in_range && t < p.T;
    float y[8];
    float amax = 0.f;
    if (real) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)t * p.H + h) * d + c * 8));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        const float2* tab = p.rope + (size_t)(p.pos0 + t) * (d / 2) + c * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 cs = __ldg(tab + e);
            rope_pair(bf16_lo(ws[e]), bf16_hi(ws[e]), cs.x, cs.y, y[2 * e], y[2 * e + 1]);
            amax = fmaxf(amax, fmaxf(fabsf(y[2 * e]), fabsf(y[2 * e + 1])));
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
    }
    // amax over the tpr lanes of this row (contiguous lanes of one warp)
    for (int off = tpr / 2; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float inv = inv_of(amax);
    uint32_t lo = e4m3x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) | (e4m3x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 16);
    uint32_t hi = e4m3x2(__fmul_rn(y[4], inv), __fmul_rn(y[5], inv)) | (e4m3x2(__fmul_rn(y[6], inv), __fmul_rn(y[7], inv)) << 16);
    if (in_range) {
        *reinterpret_cast<uint2*>(p.q8 + ((size_t)h * p.Tstride + t) * d + c * 8) = make_uint2(lo, hi);
        if (c == 0) p.qamax[(size_t)h * p.Tstride + t] = amax;
    }
}

cudaError_t launch_qprep(const QPrepParams& p, cudaStream_t s) {
    const int rows_per_block = 128 / (p.d / 8);
    const int rows = p.H * p.Tpad;
    qprep_kernel<<<(rows + rows_per_block - 1) / rows_per_block, 128, 0, s>>>(p);
    return cudaGetLastError();
}

// ============================================================== K4: attention
template <int D>
struct AttendSmem {
    static constexpr int kQ = 128 * D;            // Q tile, e4m3
    static constexpr int kK = 128 * D;            // K tile, e4m3 (per stage)
    static constexpr int kV = D * 128;            // V tile [d][128 slots], e4m3 (per stage)
    static constexpr int kV16 = D * 128 * 2;      // V tile widened to fp16: 2 K-blocks of [D][64]
    static constexpr int kP16 = 128 * 128 * 2;    // P fp16: 2 K-blocks of [128][64]
    static constexpr int offQ = 0;
    static constexpr int offK = offQ + kQ;
    static constexpr int offV = offK + 2 * kK;
    static constexpr int offV16 = offV + 2 * kV;
    static constexpr int offP16 = offV16 + kV16;
    static constexpr int offCol = offP16 + kP16;               // float colK[2][128], colV[2][128]
    static constexpr int offBar = offCol + 4 * 128 * 4;        // 8 mbarriers
    static constexpr int offMisc = offBar + 8 * 8;             // tmem addr, flag, reductions
    static constexpr int kBytes = offMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;               // slack for 1024-byte alignment
};

enum : int { kBarQ = 0, kBarKV0 = 1, kBarKV1 = 2, kBarS = 3, kBarO = 4, kBarDrain = 5 };
enum : int { kWaitQ = 1, kWaitKV = 2, kWaitS = 3, kWaitO = 4, kWaitFinal = 5 };

__device__ __forceinline__ void record_timeout(int* err, int site) {
    if (atomicCAS(err, 0, KVRING_ETIMEOUT) == 0) {
        err[1] = kKernelAttend;
        err[2] = site;
        err[3] = (int)blockIdx.x;
    }
}

template <int D>
__global__ void __launch_bounds__(128, 1)
attend_kernel(const __grid_constant__ AttendParams p, const __grid_constant__ AttendMaps maps) {
    using L = AttendSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::offQ;
    uint8_t* sK = smem + L::offK;
    uint8_t* sV = smem + L::offV;
    uint8_t* sV16 = smem + L::offV16;
    uint8_t* sP16 = smem + L::offP16;
    float* sColK = reinterpret_cast<float*>(smem + L::offCol);
    float* sColV = sColK + 256;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + L::offMisc);
    float* sRed = reinterpret_cast<float*>(smem + L::offMisc + 16);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- unit of work
    int unit = blockIdx.x;
    const int split = unit % p.splits;
    unit /= p.splits;
    const int qt = unit % p.qtiles;
    const int h = unit / p.qtiles;
    const int j0 = split * p.tiles_per_split;
    const int j1 = min(p.ntiles, j0 + p.tiles_per_split);
    const int nt = j1 - j0;
    const int zrow = p.layer * p.H + h;          // (layer, head) row of the ring tensor maps

    if (warp == 0) tmem_alloc(sTmem, 256);
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
        fence_mbar_init();
        prefetch_tmap(&maps.q8);
        prefetch_tmap(&maps.k8);
        prefetch_tmap(&maps.vt8);
    }

    // V scale reference: largest V scale among this split's valid slots
    const float* vam = p.vamax + (size_t)h * p.Rpad;
    const float* kam = p.kamax + (size_t)h * p.Rpad;
    const int s_end = min(j1 * 128, p.count);
    float svmax = 0.f;
    for (int s = j0 * 128 + tid; s < s_end; s += 128) svmax = fmaxf(svmax, scale_of(__ldg(vam + s)));
#pragma unroll
    for (int off = 16; off; off >>= 1) svmax = fmaxf(svmax, __shfl_xor_sync(0xffffffffu, svmax, off));
    if (lane == 0) sRed[warp] = svmax;

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const float sv_ref = fmaxf(fmaxf(sRed[0], sRed[1]), fmaxf(sRed[2], sRed[3]));
    const float inv_sv_ref = __frcp_rn(sv_ref);
    const uint32_t tmem = *sTmem;
    const uint32_t tS = tmem;                     // columns [0, 128): S, fp32
    const uint32_t tO = tmem + 128;               // columns [128, 128 + D): O, fp32
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    // row constants: a = (Q row scale) * log2(e) / sqrt(d)
    const int qrow = qt * 128 + tid;
    const float qa = __ldg(p.qamax + (size_t)h * p.Tstride + qrow);
    const float a = scale_of(qa) * p.log2e_rsqrt_d;

    // producer state (thread 0 only)
    int issued[2] = {0, 0}, consumed[2] = {0, 0};
    bool q_pending = false;
    auto issue_kv = [&](int stage, int j) {
        if (j == p.skip_tile) return;             // testing aid: leave this load out
        uint64_t* bar = &bars[kBarKV0 + stage];
        mbar_expect_tx(bar, (uint32_t)(L::kK + L::kV));
        tma_load_3d(sK + stage * L::kK, &maps.k8, bar, 0, j * 128, zrow);
        tma_load_3d(sV + stage * L::kV, &maps.vt8, bar, j * 128, 0, zrow);
        issued[stage]++;
    };
    if (tid == 0) {
        mbar_expect_tx(&bars[kBarQ], (uint32_t)L::kQ);
        tma_load_3d(sQ, &maps.q8, &bars[kBarQ], 0, qt * 128, h);
        q_pending = true;
        for (int st = 0; st < 2 && st < nt; ++st) issue_kv(st, j0 + st);
    }

    constexpr uint32_t idS = make_idesc(128, 128);
    constexpr uint32_t idO = make_idesc(128, D);
    const uint32_t aQ = smem_u32(sQ);
    const uint32_t aK = smem_u32(sK);
    const uint32_t aP = smem_u32(sP16);
    const uint32_t aV16 = smem_u32(sV16);

    float m_run = -INFINITY;
    float l_run = 0.f;
    bool aborted = false;

    for (int it = 0; it < nt; ++it) {
        const int stage = it & 1;
        const int j = j0 + it;
        // per-slot scales of this tile (slots past count are masked below)
        {
            const int s = j * 128 + tid;
            const bool valid = s < p.count;
            sColK[stage * 128 + tid] = valid ? scale_of(__ldg(kam + s)) : 0.f;
            sColV[stage * 128 + tid] = valid ? __fmul_rn(scale_of(__ldg(vam + s)), inv_sv_ref) : 0.f;
        }
        // S = Q K^T
        bool issue_failed = false;
        if (tid == 0) {
            bool ok = true;
            if (q_pending) {
                ok = mbar_wait(&bars[kBarQ], 0, p.timeout_ns);
                if (ok) q_pending = false; else record_timeout(p.err, kWaitQ);
            }
            if (ok) {
                ok = mbar_wait(&bars[kBarKV0 + stage], (uint32_t)(consumed[stage] & 1), p.timeout_ns);
                if (ok) consumed[stage]++; else record_timeout(p.err, kWaitKV);
            }
            if (ok) {
                tc_fence_after();
                const uint32_t aKs = aK + stage * L::kK;
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
                    mma_f8(tS, make_sdesc(aQ + k * 32, D), make_sdesc(aKs + k * 32, D), idS, k > 0 ? 1u : 0u);
                mma_commit(&bars[kBarS]);
            } else {
                issue_failed = true;
            }
        }
        // block-uniform abort decision
        if (__syncthreads_or(issue_failed)) { aborted = true; break; }

        bool ok = mbar_wait(&bars[kBarS], (uint32_t)(it & 1), p.timeout_ns);
        if (!ok) record_timeout(p.err, kWaitS);
        if (ok && it > 0) {
            ok = mbar_wait(&bars[kBarO], (uint32_t)((it - 1) & 1), p.timeout_ns);
            if (!ok) record_timeout(p.err, kWaitO);
        }
        const bool wait_failed = !ok;
        tc_fence_after();

        // widen the V tile to fp16 (exact): [D rows][128 slots] e4m3 -> 2 K-blocks of [D][64] fp16
        {
            const uint8_t* src = sV + stage * L::kV;
#pragma unroll
            for (int q = tid; q < D * 8; q += 128) {
                const int dd = q >> 3, c = q & 7;
                const uint4 w = *reinterpret_cast<const uint4*>(src + dd * 128 + ((c ^ (dd & 7)) << 4));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                uint32_t h16[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(ws[e] & 0xFFFFu), __NV_E4M3);
                    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(ws[e] >> 16), __NV_E4M3);
                    h16[2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
                    h16[2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
                }
                uint8_t* dblk = sV16 + (c >> 2) * (D * 128) + dd * 128;
                const int cb = (c & 3) * 2;
                *reinterpret_cast<uint4*>(dblk + (((cb + 0) ^ (dd & 7)) << 4)) = make_uint4(h16[0], h16[1], h16[2], h16[3]);
                *reinterpret_cast<uint4*>(dblk + (((cb + 1) ^ (dd & 7)) << 4)) = make_uint4(h16[4], h16[5], h16[6], h16[7]);
            }
        }

        // softmax on row tid
        const int nvalid = min(128, p.count - j * 128);
        const float* colK = sColK + stage * 128;
        const float* colV = sColV + stage * 128;
        float mt = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            tmem_ld32(tS + lane_off + cc * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int col = cc * 32 + e;
                if (col < nvalid) mt = fmaxf(mt, __uint_as_float(r[e]) * colK[col]);
            }
        }
        // Lazy rescale: move the running max only when it grows by more than 2^8.
        // tcgen05.ld/st are warp-collective, so a warp rescales if any of its rows
        // needs it; the other rows multiply by 1.
        const bool first = m_run == -INFINITY;
        const bool grow = !first && (mt - m_run) * a > 8.f;
        if (__any_sync(0xffffffffu, grow)) {
            const float alpha = grow ? ex2_approx((m_run - mt) * a) : 1.f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(tO + lane_off + cc * 32, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                tmem_st32(tO + lane_off + cc * 32, r);
            }
            tmem_wait_st();
            l_run *= alpha;
        }
        if (first || grow) m_run = mt;
        const float ma = m_run * a;
        float lsum = 0.f;
        uint8_t* prow = sP16 + tid * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            tmem_ld32(tS + lane_off + cc * 32, r);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const int col = cc * 32 + e;
                float p0 = 0.f, p1 = 0.f;
                if (col < nvalid) p0 = ex2_approx(fmaf(__uint_as_float(r[e]) * colK[col], a, -ma));
                if (col + 1 < nvalid) p1 = ex2_approx(fmaf(__uint_as_float(r[e + 1]) * colK[col + 1], a, -ma));
                lsum += p0 + p1;
                __half2 hv = __floats2half2_rn(p0 * colV[col], p1 * colV[col + 1]);
                pk[e / 2] = *reinterpret_cast<uint32_t*>(&hv);
            }
            uint8_t* blk = prow + (cc >> 1) * (128 * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int cb = (cc & 1) * 4 + q;
                *reinterpret_cast<uint4*>(blk + ((cb ^ (tid & 7)) << 4)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
        l_run += lsum;

        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(wait_failed)) { aborted = true; break; }
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * (128 * 128) + (k & 3) * 32;
                const uint32_t offv = (k >> 2) * (D * 128) + (k & 3) * 32;
                mma_f16(tO, make_sdesc(aP + off, 128), make_sdesc(aV16 + offv, 128), idO,
                        (it > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&bars[kBarO]);
            if (it + 2 < nt) issue_kv(stage, j0 + it + 2);
        }
    }

    if (!aborted) {
        bool ok = mbar_wait(&bars[kBarO], (uint32_t)((nt - 1) & 1), p.timeout_ns);
        if (!ok) { record_timeout(p.err, kWaitFinal); aborted = true; }
        tc_fence_after();
        // every lane reads its TMEM row (warp-collective); only real rows are stored
        const int t = qt * 128 + tid;
        const bool store = ok && t < p.T;
        const bool direct = p.splits == 1;
        const float f = direct ? sv_ref / l_run : sv_ref;
        const size_t prow_i = ((size_t)split * p.H + h) * p.Tstride + t;
        float* dst = direct ? p.out + ((size_t)t * p.H + h) * D : p.part_o + prow_i * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(tO + lane_off + cc * 32, r);
            if (store) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + cc * 32 + e) =
                        make_float4(__uint_as_float(r[e]) * f, __uint_as_float(r[e + 1]) * f,
                                    __uint_as_float(r[e + 2]) * f, __uint_as_float(r[e + 3]) * f);
            }
        }
        if (store && !direct) *reinterpret_cast<float2*>(p.part_ml + prow_i * 2) = make_float2(m_run * a, l_run);
    }
    if (aborted && tid == 0) {
        // drain: every MMA this thread issued, then every TMA copy still in flight
        mma_commit(&bars[kBarDrain]);
        mbar_wait(&bars[kBarDrain], 0, p.timeout_ns);
        if (q_pending) mbar_wait(&bars[kBarQ], 0, p.timeout_ns);
        for (int st = 0; st < 2; ++st)
            while (consumed[st] < issued[st]) {
                mbar_wait(&bars[kBarKV0 + st], (uint32_t)(consumed[st] & 1), p.timeout_ns);
                consumed[st]++;
            }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

size_t attend_smem_bytes(int d) {
    return d == 128 ? (size_t)AttendSmem<128>::kAlloc : (size_t)AttendSmem<64>::kAlloc;
}

cudaError_t launch_attend(const AttendParams& p, const AttendMaps& maps, cudaStream_t s) {
    const int grid = p.H * p.qtiles * p.splits;
    if (p.d == 128) {
        const int smem = AttendSmem<128>::kAlloc;
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attend_kernel<128><<<grid, 128, smem, s>>>(p, maps);
    } else {
        const int smem = AttendSmem<64>::kAlloc;
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attend_kernel<64><<<grid, 128, smem, s>>>(p, maps);
    }
    return cudaGetLastError();
}

// ============================================================== K5: combine splits
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, with M = max_s m_s (log2 units).
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ CombineParams p) {
    const int d = p.d;
    const int tpr = d / 4;                        // threads per row, float4 each
    const int rows_per_block = 128 / tpr;
    const int row = blockIdx.x * rows_per_block + threadIdx.x / tpr;   // over T * H, token-major
    const int c = threadIdx.x % tpr;
    if (row >= p.T * p.H) return;
    const int t = row / p.H, h = row % p.H;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s)
        M = fmaxf(M, p.part_ml[(((size_t)s * p.H + h) * p.Tstride + t) * 2]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    for (int s = 0; s < p.splits; ++s) {
        const size_t pr = ((size_t)s * p.H + h) * p.Tstride + t;
        const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + pr * 2);
        const float w = ex2_approx(ml.x - M);
        lsum += w * ml.y;
        const float4 o = *reinterpret_cast<const float4*>(p.part_o + pr * d + c * 4);
        acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
    const float inv = 1.f / lsum;
    *reinterpret_cast<float4*>(p.out + ((size_t)t * p.H + h) * d + c * 4) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
    const int rows_per_block = 128 / (p.d / 4);
    const int rows = p.T * p.H;
    combine_kernel<<<(rows + rows_per_block - 1) / rows_per_block, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvring_impl
