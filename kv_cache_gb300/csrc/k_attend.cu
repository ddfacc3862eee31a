// K3 (Q prep) and K4 (FP8 attention over the ring, with the KV-split merge).
//
// The pages have every attention call read a cache of 5,788 slots of which 757
// are new, 240 calls per step (wechild.cn news item on Runway's real-time
// Characters inference paper, paragraph 6; ai.info, "Characters funziona in
// tempo reale su quattro H100", section "La gestione della cache spostata al
// momento della scrittura"), and name the missing piece on Blackwell: an FP8
// attention kernel that accepts per-head scales (same article, section "Latenza
// dei turni e altre configurazioni GPU").
//
// K4 is one CTA of 16 warps per (head, pair of 128-row query tiles, KV split):
//  * Q (e4m3, from K3), K tiles [128 slots][d], V tiles [d][128 slots] (e4m3) and
//    the tile's K/V chunk amax rows arrive by TMA into shared memory, 3 stages.
//  * S = Q K^T runs on tcgen05 (kind::f8f6f4, M = 128, N = 64 per half tile)
//    into tensor memory, two S buffers per query tile.
//  * Thread i of a softmax warp group owns query row i (tensor-memory lane i):
//    the weight of slot c is 2^z with z = S * ks_c * a + lg2(sv_c) (K and V scale
//    of the slot's chunk, a = Q scale of the row * log2(e) / sqrt(d)).  A first
//    pass over the split's slots finds the exact row max M of z; the second
//    writes P = 2^(z - M) <= 1 as fp16 over S and sums l = sum P / sv.
//  * The V tile is widened from e4m3 to fp16 in shared memory (exact, as
//    V * 2^-8) and O += P V runs on tcgen05 (kind::f16, M = 128, N = d, P from
//    tensor memory); out = 2^8 O / l, or (2^8 O, M, l) per split for the merge.
//  * The KV splits of a (head, query pair) merge in one of three ways, chosen
//    on the host: as one thread-block cluster, reading each other's (O, M, l)
//    from distributed shared memory, when every cluster fits on the device at
//    once; else, with every CTA resident (cooperative launch), each split
//    merging a share of the rows from the others' partials in global memory;
//    else the last split to finish merging all rows.
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
    // This grid may have started before the one ahead of it finished, so it
    // waits for it before reading anything.  Only then may the attention grid
    // that follows start: that grid loads its first K/V tiles before its own
    // wait, so the ring must be final (the write ahead of this grid complete)
    // by the time any of its blocks exists.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Launched with programmatic stream serialisation (its launch overlaps the tail
// of the grid before it; it waits for that grid before reading anything).
cudaError_t launch_qprep(const QPrepParams& p, cudaStream_t s) {
    const int rows_per_block = 128 / (p.d / 8);
    const int rows = p.H * p.Tpad;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((rows + rows_per_block - 1) / rows_per_block), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qprep_kernel, p);
}



// ============================================================== K4: attention
// One CTA of 16 warps per (head, pair of 128-row query tiles, KV split):
//   warps 0-3   softmax for query tile 0 (tensor-memory lanes 0-127 of S0, O0)
//   warps 4-7   softmax for query tile 1 (S1, O1)
//   warps 8-11  per stage: the scale summaries of its four 32-column groups; in
//               the second pass also V e4m3 -> fp16 (bit operations, V * 2^-8)
//   warp 12     TMA producer (the query tiles once, then the split's tiles
//               twice: K for the first pass, K and V for the second)
//   warps 13-14 tcgen05 issuers, one per query tile
//   warp 15     idle (it keeps two softmax warps and two others on every SM
//               sub-partition, which the register split needs)
// Tensor memory (512 columns): per query tile q two S buffers of 64 columns,
// [128q, 128q + 64) and [128q + 64, 128q + 128), then O0 [256, 256 + d) and
// O1 [384, 384 + d).  A 128-slot tile is worked as two halves, half u in S
// buffer u % 2: while the softmax works on one half, S of the next is already
// in the other buffer.  In the second pass the issuer puts S_q(u + 2) right
// behind O_q += P_q(u) V in the tensor pipe, so S never overwrites P before it
// is read.  Hand-offs are mbarriers; every wait is bounded and gives up as soon
// as another warp has recorded a time-out.
template <int D>
struct AttendSmem {
    static constexpr int kStages = 3;
    static constexpr int kQ = 128 * D;            // one query tile, e4m3
    static constexpr int kK = 128 * D;            // K tile [128 slots][D], e4m3
    static constexpr int kV = D * 128;            // V tile [D][128 slots], e4m3
    static constexpr int kV16 = D * 128 * 2;      // V tile in fp16: 2 K-blocks of [D][64]
    static constexpr int offQ = 0;
    static constexpr int offK = offQ + 2 * kQ;
    static constexpr int offV = offK + kStages * kK;
    static constexpr int offV16 = offV + kStages * kV;
    // the tile's K and V chunk amax rows (fp32, 512 bytes each), then the four
    // groups' scale summaries (GroupInfo, 32 bytes each)
    static constexpr int kAmRows = 2 * 128 * 4;
    static constexpr int kAm = kAmRows + 4 * 32;
    static constexpr int offAm = offV16 + 2 * kV16;
    static constexpr int offBar = offAm + kStages * kAm;
    static constexpr int kBars = 33;
    static constexpr int offMisc = offBar + kBars * 8;
    static constexpr int kBytes = offMisc + 64;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

// mbarrier slots ([q][b]: per query tile q and S buffer b, in that order)
enum : int {
    kBQ = 0,        // query tiles landed (TMA)
    kBKVF = 1,      // [3] stage full: K, V and the amax rows (TMA)
    kBKVE = 4,      // [3] stage free: one arrival per converter warp and per softmax warp (end of its tile)
    kBSF = 7,       // [2][2] S_q half b computed (commit)
    kBPF = 11,      // [2][2] first pass: S_q half b read out; second: P_q half b written (one arrival per softmax warp)
    kBVF = 15,      // [2] fp16 V buffer full (one arrival per converter warp)
    kBVE = 17,      // [2] fp16 V buffer free (one commit per active issuer)
    kBOF = 19,      // [2] O_q complete: the last O_q += P V (commit)
    kBDrain = 21,   // drain after an abort (one commit per active issuer)
    kBIF = 22,      // [3] the stage's group summaries written (one arrival per converter warp)
    kBSF1 = 25,     // [2][2] first pass: S_q of a full tile in buffer b computed (commit)
    kBPF1 = 29,     // [2][2] first pass: that S read out (one arrival per softmax warp)
};
enum : int { kWaitQ = 1, kWaitKVFull = 2, kWaitKVEmpty = 3, kWaitS = 4, kWaitP = 5, kWaitO = 6, kWaitV16Full = 7,
             kWaitV16Empty = 8, kWaitMerge = 9 };
constexpr int kAttendThreads = 512;
constexpr int kMaxSplits = 4;   // KV splits per (head, query pair); the merge holds them all in registers

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Warp-collective bounded wait: every lane polls the same barrier word with
// the same instruction, so all see the same state and the warp never diverges
// (a divergent single-lane poll plus a broadcast costs several hundred cycles
// even when the phase is already complete).  Gives up when the phase does not
// complete within timeout_ns (and then records the time-out and raises the
// CTA's abort flag) or when the abort flag is raised.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const AttendParams& p, int site) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_test_wait(bar, parity)) return true;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
        if (__any_sync(0xffffffffu, (long long)(globaltimer_ns() - t0) > p.timeout_ns)) {
            if ((threadIdx.x & 31) == 0) {
                *abort_flag = 1;
                if (atomicCAS(p.err, 0, KVRING_ETIMEOUT) == 0) {
                    p.err[1] = kKernelAttend;
                    p.err[2] = site;
                    p.err[3] = (int)blockIdx.x;
                }
            }
            __syncwarp();
            return false;
        }
    }
}

// One arrival for the whole warp (elected lane; the warp must be converged).
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

template <int D>
__device__ __forceinline__ void issue_s_full(uint32_t tS, uint32_t aQ, uint32_t aK) {
    constexpr uint32_t id = make_idesc(128, 128);
#pragma unroll
    for (int k = 0; k < D / 32; ++k)
        mma_f8_warp(tS, make_sdesc(aQ + k * 32, D), make_sdesc(aK + k * 32, D), id, k > 0 ? 1u : 0u);
}

// S for one half tile: S[128 query rows][64 slots] = Q K_half^T, e4m3 operands in
// shared memory (K-major rows of D bytes), fp32 accumulator in tensor memory.
template <int D>
__device__ __forceinline__ void issue_s_half(uint32_t tS, uint32_t aQ, uint32_t aK) {
    constexpr uint32_t id = make_idesc(128, 64);
#pragma unroll
    for (int k = 0; k < D / 32; ++k)
        mma_f8_warp(tS, make_sdesc(aQ + k * 32, D), make_sdesc(aK + k * 32, D), id, k > 0 ? 1u : 0u);
}

// O += P V for one half tile (64 slots): P (fp16) in tensor memory at tP, 8 columns
// per 16-slot step; V fp16 in shared memory, one K-block of [D][64].
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t tO, uint32_t tP, uint32_t aV16blk, bool accumulate) {
    constexpr uint32_t id = make_idesc(128, D);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        mma_f16_ts_warp(tO, tP + k * 8, make_sdesc(aV16blk + k * 32, 128), id, (accumulate || k > 0) ? 1u : 0u);
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

constexpr float kInv448 = 1.f / 448.f;

// Largest of 32 raw scores.
__device__ __forceinline__ float max32(const uint32_t (&r)[32]) {
    float m0 = fmax3(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]));
    float m1 = fmax3(__uint_as_float(r[3]), __uint_as_float(r[4]), __uint_as_float(r[5]));
    float m2 = fmax3(__uint_as_float(r[6]), __uint_as_float(r[7]), __uint_as_float(r[8]));
    float m3 = fmax3(__uint_as_float(r[9]), __uint_as_float(r[10]), __uint_as_float(r[11]));
#pragma unroll
    for (int e = 12; e < 28; e += 8) {
        m0 = fmax3(m0, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
        m1 = fmax3(m1, __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        m2 = fmax3(m2, __uint_as_float(r[e + 4]), __uint_as_float(r[e + 5]));
        m3 = fmax3(m3, __uint_as_float(r[e + 6]), __uint_as_float(r[e + 7]));
    }
    m0 = fmax3(m0, __uint_as_float(r[28]), __uint_as_float(r[29]));
    m1 = fmax3(m1, __uint_as_float(r[30]), __uint_as_float(r[31]));
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// One-range group: P = 2^(raw * c1 + c0) packed as fp16 pairs.  Returns the
// group's share of the row sum, (sum of the fp32 P + fp16 rounding of the
// largest one) * inv_sv; graw is the group's largest raw score.
__device__ __forceinline__ float p_one_range(const uint32_t (&r)[32], float c1, float c0, float graw, float inv_sv,
                                             uint32_t (&pk)[16]) {
    const float2 c1v = make_float2(c1, c1), c0v = make_float2(c0, c0);
    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        const float2 x01 = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c1v, c0v);
        const float2 x23 = ffma2(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), c1v, c0v);
        const float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
        const float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
        pk[e / 2] = h2_bits(__floats2half2_rn(p01.x, p01.y));
        pk[e / 2 + 1] = h2_bits(__floats2half2_rn(p23.x, p23.y));
        s0 = fadd2(s0, p01);
        s1 = fadd2(s1, p23);
    }
    const float pm = ex2_approx(fmaf(graw, c1, c0));
    const float corr = __half2float(__float2half_rn(pm)) - pm;
    return ((s0.x + s0.y) + (s1.x + s1.y) + corr) * inv_sv;
}

// Scales of one 32-column group of a tile, for the general (not one-range) path.
// Lane e's own column is 32g + e.  kind 0: one range; 1: range A = columns
// [0, b), range B = [b, 32); 2: per-column scales.  k* already carry the row's a.
struct GroupScales {
    int kind, b;
    float kA, lA, iA, kB, lB, iB;   // ks * a, lg2(sv), 1 / sv of ranges A and B
    float ks, ls, is;               // ks, lg2(sv), 1 / sv of the lane's own column (kind 2 only)
};

// Scale summary of one 32-column group of a tile, written once per tile by the
// converter warps and read by all softmax warps.
struct GroupInfo {
    float ks, ls, is;      // range A: K scale, lg2(V scale), 1 / V scale (0, -inf, 0 past the valid slots)
    int kind_b;            // kind | b << 8
    float ksB, lsB, isB;   // range B
    float pad;
};

// The K/V scales of column 32g + lane; ka / va are -1 past the valid slots.
__device__ __forceinline__ void column_scales(const float* am, int col, bool valid, float& ka, float& va, float& ks,
                                              float& ls, float& is) {
    ka = valid ? am[col] : -1.f;
    va = valid ? am[128 + col] : -1.f;
    const float sv = va == 0.f ? 1.f : va * kInv448;
    ks = valid ? (ka == 0.f ? 1.f : ka * kInv448) : 0.f;
    ls = valid ? lg2_approx(sv) : -INFINITY;
    is = valid ? rcp_approx(sv) : 0.f;
}

// Builds the summary of group g (one warp, lane = column within the group); lane
// 0 writes it.
__device__ __forceinline__ void write_group_info(const float* am, int g, int slot0, int count, int lane,
                                                 GroupInfo* out) {
    const int col = g * 32 + lane;
    float ka, va, ks, ls, is;
    column_scales(am, col, slot0 + col < count, ka, va, ks, ls, is);
    const float ka0 = __shfl_sync(0xffffffffu, ka, 0);
    const float va0 = __shfl_sync(0xffffffffu, va, 0);
    const uint32_t diff = __ballot_sync(0xffffffffu, ka != ka0 || va != va0);
    int kind = 0, b = 32;
    if (diff) {
        b = __ffs(diff) - 1;
        const float kab = __shfl_sync(0xffffffffu, ka, b);
        const float vab = __shfl_sync(0xffffffffu, va, b);
        kind = __ballot_sync(0xffffffffu, lane >= b && (ka != kab || va != vab)) ? 2 : 1;
    }
    const float ksA = __shfl_sync(0xffffffffu, ks, 0), lsA = __shfl_sync(0xffffffffu, ls, 0);
    const float isA = __shfl_sync(0xffffffffu, is, 0);
    const int bs = b & 31;
    const float ksB = __shfl_sync(0xffffffffu, ks, bs), lsB = __shfl_sync(0xffffffffu, ls, bs);
    const float isB = __shfl_sync(0xffffffffu, is, bs);
    if (lane == 0) {
        float4* o = reinterpret_cast<float4*>(out);
        o[0] = make_float4(ksA, lsA, isA, __int_as_float(kind | (b << 8)));
        o[1] = make_float4(ksB, lsB, isB, 0.f);
    }
}

// General-path scales of group g from its summary (and, for per-column groups,
// from the amax rows).
__device__ __forceinline__ GroupScales group_scales(const GroupInfo* info, const float* am, int g, int slot0,
                                                    int count, float a, int lane) {
    GroupScales s;
    const float4 i0 = reinterpret_cast<const float4*>(info + g)[0];
    const float4 i1 = reinterpret_cast<const float4*>(info + g)[1];
    const int kb = __float_as_int(i0.w);
    s.kind = kb & 3;
    s.b = kb >> 8;
    s.kA = i0.x * a;
    s.lA = i0.y;
    s.iA = i0.z;
    s.kB = i1.x * a;
    s.lB = i1.y;
    s.iB = i1.z;
    s.ks = s.ls = s.is = 0.f;
    if (s.kind == 2) {
        const int col = g * 32 + lane;
        float ka, va;
        column_scales(am, col, slot0 + col < count, ka, va, s.ks, s.ls, s.is);
    }
    return s;
}

// Row max of z = raw * ks * a + lg2(sv) over one group, general path.
__device__ __forceinline__ float zmax_group(const uint32_t (&r)[32], const GroupScales& s, float a) {
    if (s.kind == 0) return fmaf(max32(r), s.kA, s.lA);
    float m = -INFINITY;
    if (s.kind == 1) {
        float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float x = __uint_as_float(r[e]);
            mA = fmaxf(mA, e < s.b ? x : -INFINITY);
            mB = fmaxf(mB, e < s.b ? -INFINITY : x);
        }
        return fmaxf(fmaf(mA, s.kA, s.lA), fmaf(mB, s.kB, s.lB));
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float ksa = __shfl_sync(0xffffffffu, s.ks, e) * a;
        const float ls = __shfl_sync(0xffffffffu, s.ls, e);
        m = fmaxf(m, fmaf(__uint_as_float(r[e]), ksa, ls));
    }
    return m;
}

// P of one group, general path (kinds 1 and 2 sum the rounded P themselves).
__device__ __forceinline__ float p_group(const uint32_t (&r)[32], const GroupScales& s, float M, float a,
                                         uint32_t (&pk)[16]) {
    if (s.kind == 0) return p_one_range(r, s.kA, s.lA - M, max32(r), s.iA, pk);
    float lsum = 0.f;
    if (s.kind == 1) {
        const float c0A = s.lA - M, c0B = s.lB - M;
        float sA = 0.f, sB = 0.f;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            const bool a0 = e < s.b, a1 = e + 1 < s.b;
            const float p0 = ex2_approx(fmaf(__uint_as_float(r[e]), a0 ? s.kA : s.kB, a0 ? c0A : c0B));
            const float p1 = ex2_approx(fmaf(__uint_as_float(r[e + 1]), a1 ? s.kA : s.kB, a1 ? c0A : c0B));
            const __half2 hv = __floats2half2_rn(p0, p1);
            pk[e / 2] = h2_bits(hv);
            const float2 back = __half22float2(hv);
            sA += (a0 ? back.x : 0.f) + (a1 ? back.y : 0.f);
            sB += (a0 ? 0.f : back.x) + (a1 ? 0.f : back.y);
        }
        return sA * s.iA + sB * s.iB;
    }
    // per-column scales (slots past the valid count have ks = 0, lg2 sv = -inf,
    // hence P exactly 0; the exponent is capped so that 2^x stays finite)
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const float k0 = __shfl_sync(0xffffffffu, s.ks, e) * a, k1 = __shfl_sync(0xffffffffu, s.ks, e + 1) * a;
        const float l0 = __shfl_sync(0xffffffffu, s.ls, e), l1 = __shfl_sync(0xffffffffu, s.ls, e + 1);
        const float i0 = __shfl_sync(0xffffffffu, s.is, e), i1 = __shfl_sync(0xffffffffu, s.is, e + 1);
        const float p0 = ex2_approx(fminf(fmaf(__uint_as_float(r[e]), k0, l0 - M), 64.f));
        const float p1 = ex2_approx(fminf(fmaf(__uint_as_float(r[e + 1]), k1, l1 - M), 64.f));
        const __half2 hv = __floats2half2_rn(p0, p1);
        pk[e / 2] = h2_bits(hv);
        const float2 back = __half22float2(hv);
        lsum = fmaf(back.x, i0, fmaf(back.y, i1, lsum));
    }
    return lsum;
}

// The general paths (a group that is not one range) are rare -- a chunk boundary
// or the ring's last valid slot falls inside the group -- and large once unrolled,
// so each has one out-of-line copy that reloads the group's 32 scores from tensor
// memory itself: the hot loop stays small in the instruction cache and no
// register array crosses the call.
__device__ __noinline__ float zmax_general(uint32_t taddr, const GroupInfo* info, const float* am, int g, int slot0,
                                           int count, float a, int lane) {
    uint32_t r[32];
    tmem_ld32_async(taddr, r);
    tmem_wait_ld_dep(r);
    return zmax_group(r, group_scales(info, am, g, slot0, count, a, lane), a);
}

// P of group g read from tsrc, stored as 16 packed fp16 columns at tdst; returns
// the group's share of the row sum.
__device__ __noinline__ float p_general(uint32_t tsrc, uint32_t tdst, const GroupInfo* info, const float* am, int g,
                                        int slot0, int count, float a, float M, int lane) {
    uint32_t r[32], pk[16];
    tmem_ld32_async(tsrc, r);
    tmem_wait_ld_dep(r);
    const float l = p_group(r, group_scales(info, am, g, slot0, count, a, lane), M, a, pk);
    tmem_st16(tdst, pk);
    return l;
}

template <int D>
__global__ void __launch_bounds__(kAttendThreads, 1)
attend_kernel(const __grid_constant__ AttendParams p, const __grid_constant__ AttendMaps maps) {
    using L = AttendSmem<D>;
    constexpr int NST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + L::offQ;
    uint8_t* sK = smem + L::offK;
    uint8_t* sV = smem + L::offV;
    uint8_t* sV16 = smem + L::offV16;
    uint8_t* sAm = smem + L::offAm;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + L::offMisc);
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
    volatile int* sLast = reinterpret_cast<volatile int*>(smem + L::offMisc + 8);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // the grid after this one may be scheduled as SMs free up (it waits for this
    // one before it reads or writes anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    int u = blockIdx.x;
    const int split = u % p.splits;
    u /= p.splits;
    const int pair = u % p.npairs;
    const int h = u / p.npairs;
    const int j0 = split * p.tiles_per_split;
    const int nt = min(p.ntiles, j0 + p.tiles_per_split) - j0;
    const int nq = ((2 * pair + 1) * 128 < p.T) ? 2 : 1;
    const int zrow = p.layer * p.H + h;
    const float* kam = p.kamax + (size_t)h * p.Rpad;
    const float* vam = p.vamax + (size_t)h * p.Rpad;

    if (warp == 0) tmem_alloc(sTmem, 512);
    if (tid == 0) {
        // A stage is free again after the four converter warps (its V tile is
        // widened) and each softmax warp of each active query tile (at the end of
        // its tile: its S MMAs are done and its scale rows read).
        const int kve = 4 + 4 * nq;   // per stage: one arrival per converter warp and per softmax warp
        const int counts[L::kBars] = {1, 1, 1, 1, kve, kve, kve, 1,  1,  1,  1, 4, 4, 4, 4, 4, 4,
                                      nq, nq, 1,  1,  nq, 4, 4, 4, 1, 1, 1, 1,  4, 4, 4, 4};
        for (int b = 0; b < L::kBars; ++b) mbar_init(&bars[b], counts[b]);
        fence_mbar_init();
        *sAbort = 0;
        *sLast = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sTmem;
    const int nh = 2 * nt;   // half tiles of 64 slots in one pass over the split

    // softmax state (warps 0-7), kept for the epilogue
    const int q = warp >> 2;
    const int wq = warp & 3;
    const int row = tid & 127;
    const int qrow = (2 * pair + q) * 128 + row;
    float M = -INFINITY, l_run = 0.f;
    // producer state (warp 12, lane 0)
    int issued[NST];
#pragma unroll
    for (int st = 0; st < NST; ++st) issued[st] = 0;
    bool q_issued = false;

    // Register split.  The launch gives each of the 16 warps 128 registers per
    // thread, and every SM sub-partition (warps w, w+4, w+8, w+12) holds two
    // softmax warps and two others; 2 x 176 + 2 x 80 = 2 x 128 + 2 x 128, so the
    // increase always fits in the registers its own sub-partition released.
    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    }

    if (warp < 8) {
        // ------------------------------------------------------------ softmax
        // Weights in log2 units: slot c of row t has z = S[t][c] * ks_c * a_t + lg2(sv_c)
        // with a_t = (Q scale of the row) * log2(e) / sqrt(d), ks / sv the slot's K / V
        // scales.  The V scale rides in the exponent, so P = 2^(z - M) is the weight
        // already multiplied by the V scale (O += P V8 then sums w * sv * v8), and the
        // row sum takes it out again with 1/sv.
        // Two passes over the split's slots: the first computes S only and keeps the
        // exact row max M of z; the second computes P = 2^(z - M) <= 1 and O += P V
        // with M fixed, so O is never rescaled.  Either pass has two S buffers per
        // query tile, so that the next S is computed while this one is worked on:
        // the first pass uses full tiles in S_q and (while it is unused) O_q, the
        // second half tiles of 64 slots in the two halves of S_q.
        const bool active = q < nq;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + 128 * q + lane_off;
        const uint32_t tO = tmem + 256 + 128 * q + lane_off;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // Q prep has finished
        const float a = scale_of(__ldg(p.qamax + (size_t)h * p.Tstride + qrow)) * p.log2e_rsqrt_d;
        float gk[4], gl[4], gi[4];
        bool uni[2];
        int kinds = 0;   // 8 bits per group of the current tile: its kind (0 = one range)
        const float* am = nullptr;
        const GroupInfo* info = nullptr;
        int slot0 = 0;
        // Tile setup from the converter's group summaries of stage load ld.  The
        // columns of one chunk share one pair of scales, so a 32-column group is
        // usually one range; a half whose two groups both are (the common case)
        // takes the fast path below.
        auto tile_setup = [&](int ld) -> bool {
            const int st = ld % NST;
            slot0 = (j0 + ld % nt) * 128;
            am = reinterpret_cast<const float*>(sAm + st * L::kAm);   // K amax [128], V amax [128]
            info = reinterpret_cast<const GroupInfo*>(sAm + st * L::kAm + L::kAmRows);
            if (!warp_wait(&bars[kBIF + st], (uint32_t)((ld / NST) & 1), sAbort, p, kWaitKVFull)) return false;
            kinds = 0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 i0 = reinterpret_cast<const float4*>(info + g)[0];
                gk[g] = i0.x * a;   // a is this thread's own row's
                gl[g] = i0.y;
                gi[g] = i0.z;
                kinds |= (__float_as_int(i0.w) & 3) << (8 * g);
            }
            uni[0] = (kinds & 0xFFFF) == 0;
            uni[1] = (kinds >> 16) == 0;
            return true;
        };
        // row max of z over two one-range groups (2 hb, 2 hb + 1) held in registers
        auto zmax2 = [&](const uint32_t (&ra)[32], const uint32_t (&rb)[32], int hb) -> float {
            return fmaxf(fmaf(max32(ra), hb ? gk[2] : gk[0], hb ? gl[2] : gl[0]),
                         fmaf(max32(rb), hb ? gk[3] : gk[1], hb ? gl[3] : gl[1]));
        };
        auto one_range = [&](int g) -> bool { return ((kinds >> (8 * g)) & 3) == 0; };
        // the same when a group of the half is not one range: that group is read
        // again from tensor memory at taddr (+ 32) on the general path
        auto zmax2_mixed = [&](const uint32_t (&ra)[32], const uint32_t (&rb)[32], uint32_t taddr, int hb) -> float {
            const float za = one_range(2 * hb) ? fmaf(max32(ra), hb ? gk[2] : gk[0], hb ? gl[2] : gl[0])
                                               : zmax_general(taddr, info, am, 2 * hb, slot0, p.count, a, lane);
            const float zb = one_range(2 * hb + 1) ? fmaf(max32(rb), hb ? gk[3] : gk[1], hb ? gl[3] : gl[1])
                                                   : zmax_general(taddr + 32, info, am, 2 * hb + 1, slot0, p.count, a, lane);
            return fmaxf(za, zb);
        };
        // First pass, one full tile at a time in S buffer j % 2 (S_q or, while it is
        // unused, O_q's columns): the row max M of z.
        for (int j = 0; active && j < nt; ++j) {
            const int st = j % NST, b = j & 1;
            if (!tile_setup(j)) break;
            if (!warp_wait(&bars[kBSF1 + 2 * q + b], (uint32_t)((j >> 1) & 1), sAbort, p, kWaitS)) break;
            tc_fence_after();
            const uint32_t tSj = b ? tO : tS;
            float tz;
            {
                uint32_t ra[32], rb[32];
                tmem_ld32_async(tSj, ra);
                tmem_ld32_async(tSj + 32, rb);
                tmem_wait_ld_dep(ra);
                tmem_dep(rb);
                tz = uni[0] ? zmax2(ra, rb, 0) : zmax2_mixed(ra, rb, tSj, 0);
            }
            {
                uint32_t ra[32], rb[32];
                tmem_ld32_async(tSj + 64, ra);
                tmem_ld32_async(tSj + 96, rb);
                tmem_wait_ld_dep(ra);
                tmem_dep(rb);
                // the buffer is free again once read (the general path reads it again)
                if (uni[1]) {
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_warp(&bars[kBPF1 + 2 * q + b]);
                    tz = fmaxf(tz, zmax2(ra, rb, 1));
                } else {
                    tz = fmaxf(tz, zmax2_mixed(ra, rb, tSj + 64, 1));
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_warp(&bars[kBPF1 + 2 * q + b]);
                }
            }
            M = fmaxf(M, tz);
            // the end of the stage: its S MMAs are done and its scale rows read
            __syncwarp();
            mbar_arrive_warp(&bars[kBKVE + st]);
        }
        // Second pass, half tiles: P = 2^(z - M) <= 1 with M fixed.
        for (int u = 0; active && u < nh; ++u) {
            const int ld = nt + (u >> 1), hb = u & 1, st = ld % NST;   // ld: the stage load this half reads
            const uint32_t tSb = tS + 64 * hb;
            if (hb == 0 && !tile_setup(ld)) break;
            const bool un = uni[hb];
            const int g0 = 2 * hb;   // the half's groups are g0 and g0 + 1
            if (!warp_wait(&bars[kBSF + 2 * q + hb], (uint32_t)((u >> 1) & 1), sAbort, p, kWaitS)) break;
            tc_fence_after();
            // the half's S (two groups of 32 columns), read once into registers
            uint32_t ra[32], rb[32];
            tmem_ld32_async(tSb, ra);
            tmem_ld32_async(tSb + 32, rb);
            tmem_wait_ld_dep(ra);
            tmem_dep(rb);
            {
                // P = 2^(z - M) as fp16, written over the half's S buffer (group g of
                // the half to columns [16g, 16g + 16), which hold only values already
                // read).  The row sum must use the same (rounded) weights that
                // O += P V sees wherever one weight dominates: a one-range group sums
                // the fp32 P and adds back the fp16 rounding of its largest element
                // (the row's dominant weight is always one of them; the other
                // elements' rounding is at most 2^-12 of their own, non-dominant,
                // share); the other kinds sum the rounded values.
                float lsum;
                if (un) {
                    uint32_t pk[16];
                    lsum = p_one_range(ra, hb ? gk[2] : gk[0], (hb ? gl[2] : gl[0]) - M, max32(ra), hb ? gi[2] : gi[0], pk);
                    tmem_st16(tSb, pk);
                    lsum += p_one_range(rb, hb ? gk[3] : gk[1], (hb ? gl[3] : gl[1]) - M, max32(rb), hb ? gi[3] : gi[1], pk);
                    tmem_st16(tSb + 16, pk);
                } else {
                    // each group on its own path; group g0's P goes to columns [0, 16)
                    // before group g0 + 1 is (re)read from [32, 64)
                    uint32_t pk[16];
                    if (one_range(g0)) {
                        lsum = p_one_range(ra, hb ? gk[2] : gk[0], (hb ? gl[2] : gl[0]) - M, max32(ra), hb ? gi[2] : gi[0], pk);
                        tmem_st16(tSb, pk);
                    } else {
                        lsum = p_general(tSb, tSb, info, am, g0, slot0, p.count, a, M, lane);
                    }
                    if (one_range(g0 + 1)) {
                        lsum += p_one_range(rb, hb ? gk[3] : gk[1], (hb ? gl[3] : gl[1]) - M, max32(rb), hb ? gi[3] : gi[1], pk);
                        tmem_st16(tSb + 16, pk);
                    } else {
                        lsum += p_general(tSb + 32, tSb + 16, info, am, g0 + 1, slot0, p.count, a, M, lane);
                    }
                }
                l_run += lsum;
                // P_q(u) handed over once all 32 lanes' stores are done: one arrival per warp
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                mbar_arrive_warp(&bars[kBPF + 2 * q + hb]);
            }
            if (hb == 1) {
                // the end of the stage: its S MMAs are done and its scale rows read
                __syncwarp();
                mbar_arrive_warp(&bars[kBKVE + st]);
            }
        }
        if (active && !*sAbort) {
            // O_q is complete once the last O_q += P_q V has finished
            if (warp_wait(&bars[kBOF + q], 0u, sAbort, p, kWaitO)) tc_fence_after();
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ V e4m3 -> fp16
        // Per stage load: each converter warp summarises the scales of one 32-column
        // group (the softmax warps read the summaries); in the second pass the V tile
        // is then widened into fp16 buffer j % 2, once both issuers have committed
        // their last O += P V of tile j - 2.
        const int c0 = tid - 256;
        for (int ld = 0; ld < 2 * nt; ++ld) {
            const int st = ld % NST;
            if (!warp_wait(&bars[kBKVF + st], (uint32_t)((ld / NST) & 1), sAbort, p, kWaitKVFull)) break;
            write_group_info(reinterpret_cast<const float*>(sAm + st * L::kAm), warp - 8, (j0 + ld % nt) * 128, p.count,
                             lane, reinterpret_cast<GroupInfo*>(sAm + st * L::kAm + L::kAmRows) + (warp - 8));
            __syncwarp();
            mbar_arrive_warp(&bars[kBIF + st]);
            if (ld >= nt) {
                const int it = ld - nt, b = it & 1;
                if (it >= 2 && !warp_wait(&bars[kBVE + b], (uint32_t)(((it >> 1) - 1) & 1), sAbort, p, kWaitV16Empty))
                    break;
                const uint8_t* src = sV + st * L::kV;
                uint8_t* dst = sV16 + b * L::kV16;
#pragma unroll
                for (int qq = c0; qq < D * 8; qq += 128) {
                    const int dd = qq >> 3, c = qq & 7;
                    const uint4 w = *reinterpret_cast<const uint4*>(src + dd * 128 + ((c ^ (dd & 7)) << 4));
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    // e4m3 -> fp16 with integer operations: sign to bit 15, the other 7
                    // bits to bits 7-13, which is the fp16 code of value * 2^-8
                    // (subnormals included); the 2^8 is applied to O at the end
                    uint32_t h16[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t lo = __byte_perm(ws[e], 0u, 0x1404u);   // [0, b0, 0, b1]
                        const uint32_t hi = __byte_perm(ws[e], 0u, 0x3424u);   // [0, b2, 0, b3]
                        h16[2 * e] = (lo & 0x80008000u) | ((lo >> 1) & 0x3F803F80u);
                        h16[2 * e + 1] = (hi & 0x80008000u) | ((hi >> 1) & 0x3F803F80u);
                    }
                    uint8_t* dblk = dst + (c >> 2) * (D * 128) + dd * 128;
                    const int cb = (c & 3) * 2;
                    *reinterpret_cast<uint4*>(dblk + (((cb + 0) ^ (dd & 7)) << 4)) =
                        make_uint4(h16[0], h16[1], h16[2], h16[3]);
                    *reinterpret_cast<uint4*>(dblk + (((cb + 1) ^ (dd & 7)) << 4)) =
                        make_uint4(h16[4], h16[5], h16[6], h16[7]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_warp(&bars[kBVF + b]);
            }
            __syncwarp();
            mbar_arrive_warp(&bars[kBKVE + st]);
        }
    } else if (warp == 12) {
        // ------------------------------------------------------------ TMA producer
        // The split's tiles twice: K (and the amax rows) for the first pass, then K,
        // V and the amax rows for the second.
        if (lane == 0) {
            prefetch_tmap(&maps.q8);
            prefetch_tmap(&maps.k8);
            prefetch_tmap(&maps.vt8);
        }
        for (int ld = 0; ld < 2 * nt; ++ld) {
            if (ld == (nt < NST ? nt : NST)) {
                // the query tiles, once the first stages are on their way and Q prep
                // (the grid before this one) has finished; the stages above could
                // be issued earlier because this grid starts only after Q prep has
                // waited for the grid before it (the write of the ring)
                asm volatile("griddepcontrol.wait;" ::: "memory");
                mbar_expect_tx_warp(&bars[kBQ], (uint32_t)(nq * L::kQ));
                tma_load_3d_warp(sQ, &maps.q8, &bars[kBQ], 0, (2 * pair) * 128, h);
                if (nq == 2) tma_load_3d_warp(sQ + L::kQ, &maps.q8, &bars[kBQ], 0, (2 * pair + 1) * 128, h);
                q_issued = true;
            }
            const int st = ld % NST;
            if (ld >= NST && !warp_wait(&bars[kBKVE + st], (uint32_t)(((ld / NST) - 1) & 1), sAbort, p, kWaitKVEmpty))
                break;
            const int j = j0 + ld % nt;
            const bool second = ld >= nt;
            if (j != p.skip_tile) {
                // the whole warp issues (elected lane)
                mbar_expect_tx_warp(&bars[kBKVF + st], (uint32_t)(L::kK + L::kAmRows + (second ? L::kV : 0)));
                tma_load_3d_warp(sK + st * L::kK, &maps.k8, &bars[kBKVF + st], 0, j * 128, zrow);
                if (second) tma_load_3d_warp(sV + st * L::kV, &maps.vt8, &bars[kBKVF + st], j * 128, 0, zrow);
                bulk_g2s_warp(sAm + st * L::kAm, kam + (size_t)j * 128, 512, &bars[kBKVF + st]);
                bulk_g2s_warp(sAm + st * L::kAm + 512, vam + (size_t)j * 128, 512, &bars[kBKVF + st]);
                issued[st]++;
            }
        }
    } else if (warp == 13 || warp == 14) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 13 drives query tile 0, warp 14 query tile 1.  Half u uses S buffer
        // u % 2.  First pass: S_q(u + 2) as soon as the softmax has read S_q(u) out.
        // Second pass: O_q += P_q(u) V as soon as P_q(u) is written, then, into the
        // same buffer, S_q(u + 2); the tensor pipe runs them in that order, so S
        // never overwrites P before it is read.
        const int qq = warp - 13;
        if (qq < nq) {
            const uint32_t tSq = tmem + 128 * qq;
            const uint32_t tOq = tmem + 256 + 128 * qq;
            const uint32_t aQ = smem_u32(sQ) + qq * L::kQ;
            const uint32_t aK = smem_u32(sK);
            const uint32_t aV16 = smem_u32(sV16);
            bool ok = warp_wait(&bars[kBQ], 0, sAbort, p, kWaitQ);
            // First pass: full tiles j in buffer j % 2 (S_q, O_q); S(j + 2) as soon as
            // the softmax has read S(j) out.
            for (int j = 0; ok && j < nt + 2; ++j) {
                if (j >= 2) {
                    ok = warp_wait(&bars[kBPF1 + 2 * qq + (j & 1)], (uint32_t)(((j - 2) >> 1) & 1), sAbort, p, kWaitP);
                    if (!ok) break;
                }
                if (j >= nt) continue;
                const int st = j % NST;
                ok = warp_wait(&bars[kBKVF + st], (uint32_t)((j / NST) & 1), sAbort, p, kWaitKVFull);
                if (!ok) break;
                tc_fence_after();
                issue_s_full<D>((j & 1) ? tOq : tSq, aQ, aK + st * L::kK);
                mma_commit_warp(&bars[kBSF1 + 2 * qq + (j & 1)]);
            }
            // Second pass: half tiles u in buffer u % 2 of S_q.
            if (ok) {
                const int st = nt % NST;
                ok = warp_wait(&bars[kBKVF + st], (uint32_t)((nt / NST) & 1), sAbort, p, kWaitKVFull);
                if (ok) {
                    tc_fence_after();
                    issue_s_half<D>(tSq, aQ, aK + st * L::kK);
                    mma_commit_warp(&bars[kBSF + 2 * qq]);
                    issue_s_half<D>(tSq + 64, aQ, aK + st * L::kK + 64 * D);
                    mma_commit_warp(&bars[kBSF + 2 * qq + 1]);
                }
            }
            for (int u = 0; ok && u < nh; ++u) {
                const int it = u >> 1, hb = u & 1;   // second-pass tile of this half
                if (hb == 0) ok = warp_wait(&bars[kBVF + (it & 1)], (uint32_t)((it >> 1) & 1), sAbort, p, kWaitV16Full);
                ok = ok && warp_wait(&bars[kBPF + 2 * qq + hb], (uint32_t)(it & 1), sAbort, p, kWaitP);
                const int ldn = nt + it + 1, stn = ldn % NST;   // the stage load of half u + 2
                const bool has_next = u + 2 < nh;
                if (ok && has_next && hb == 0)
                    ok = warp_wait(&bars[kBKVF + stn], (uint32_t)((ldn / NST) & 1), sAbort, p, kWaitKVFull);
                if (!ok) break;
                tc_fence_after();
                // the whole warp issues (warp-uniform operands, one elected lane)
                issue_pv_half<D>(tOq, tSq + 64 * hb, aV16 + (it & 1) * L::kV16 + hb * (D * 128), u > 0);
                if (hb == 1) mma_commit_warp(&bars[kBVE + (it & 1)]);
                if (has_next) {
                    issue_s_half<D>(tSq + 64 * hb, aQ, aK + stn * L::kK + hb * 64 * D);
                    mma_commit_warp(&bars[kBSF + 2 * qq + hb]);
                } else if (u == nh - 1) {
                    mma_commit_warp(&bars[kBOF + qq]);
                }
            }
        }
    }

    // ---------------------------------------------------------------- join
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Back to the launch split (128 each) for the epilogue and the split merge.
    // Only after the barrier: a warp that asked for its registers back earlier
    // could take them before a softmax warp of its sub-partition had made its
    // own increase, and that increase would then never be granted.
    if (warp < 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 128;" ::: "memory");
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 128;" ::: "memory");
    }
    const bool aborted = *sAbort != 0;
    if (aborted) {
        // nothing of ours may still be in flight when the CTA goes on
        if ((warp == 13 || warp == 14) && warp - 13 < nq) {
            mma_commit_warp(&bars[kBDrain]);
            if (lane == 0) mbar_wait(&bars[kBDrain], 0, p.timeout_ns);
            __syncwarp();
        }
        if (warp == 12 && lane == 0) {
            if (q_issued) mbar_wait(&bars[kBQ], 0, p.timeout_ns);
            for (int st = 0; st < NST; ++st)
                if (issued[st] > 0) mbar_wait(&bars[kBKVF + st], (uint32_t)((issued[st] - 1) & 1), p.timeout_ns);
        }
        __syncthreads();
    }
    // ---------------------------------------------------------------- epilogue
    // Every stage is consumed (or drained), so the tiles' shared memory is free:
    // each softmax thread puts its row of O (unnormalised) and its (M, l) there,
    // and the rows then go out one warp per row (coalesced 512-byte stores):
    // normalised to out with one KV split, else as this split's partial.
    constexpr int kORow = D + 4;   // padded row of O in shared memory (fp32)
    float* sO = reinterpret_cast<float*>(smem);                            // [256][kORow]
    float2* sML = reinterpret_cast<float2*>(smem + 256 * kORow * 4);       // [256]
    if (warp < 8 && q < nq) {
        const uint32_t tO = tmem + 256 + 128 * q + ((uint32_t)(wq * 32) << 16);
        float* orow = sO + (size_t)(q * 128 + row) * kORow;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(tO + cc * 32, r);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4*>(orow + cc * 32 + e) =
                    make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                __uint_as_float(r[e + 3]));
        }
        sML[q * 128 + row] = make_float2(M, l_run);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    const int rows = nq * 128;
    const bool lanes_d = lane < D / 4;   // lane i holds output values 4i..4i+3
    if (p.splits == 1) {
        for (int rr = warp; rr < rows; rr += kAttendThreads / 32) {
            const int t = pair * 256 + rr;
            if (t >= p.T || !lanes_d) continue;
            const float f = 256.f / sML[rr].y;   // V was widened as V * 2^-8
            const float4 o = *reinterpret_cast<const float4*>(sO + (size_t)rr * kORow + 4 * lane);
            *reinterpret_cast<float4*>(p.out + ((size_t)t * p.H + h) * D + 4 * lane) =
                make_float4(o.x * f, o.y * f, o.z * f, o.w * f);
        }
        return;
    }
    constexpr int kRowsAtOnce = 4;
    if (p.cluster) {
        // The splits of this (head, pair) are the CTAs of one cluster (rank = split).
        // Once all have their O and (M, l) in shared memory, each merges its share
        // of the rows reading the others' shared memory directly: no partials in
        // global memory, no counters.  Every thread of every CTA of the cluster
        // reaches both barriers (aborted or not), so neither waits for ever.
        cluster_sync_all();
        const int r0 = split * rows / p.splits, r1 = (split + 1) * rows / p.splits;
        uint32_t o_at[kMaxSplits], ml_at[kMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp) {
            const uint32_t rank = (uint32_t)(sp < p.splits ? sp : 0);
            o_at[sp] = dsmem_map(smem_u32(sO), rank);
            ml_at[sp] = dsmem_map(smem_u32(sML), rank);
        }
        for (int rb = r0 + warp * kRowsAtOnce; rb < r1; rb += kRowsAtOnce * (kAttendThreads / 32)) {
            float2 ml[kRowsAtOnce][kMaxSplits];
            float4 o[kRowsAtOnce][kMaxSplits];
#pragma unroll
            for (int k = 0; k < kRowsAtOnce; ++k) {
                const int rr = rb + k;
                const bool mine = rr < r1 && pair * 256 + rr < p.T;
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) {
                    ml[k][sp] = make_float2(-INFINITY, 0.f);
                    o[k][sp] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (sp < p.splits && mine) {
                        ml[k][sp] = dsmem_ld_f2(ml_at[sp] + (uint32_t)rr * 8u);
                        if (lanes_d) o[k][sp] = dsmem_ld_f4(o_at[sp] + (uint32_t)(rr * kORow + 4 * lane) * 4u);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kRowsAtOnce; ++k) {
                const int t = pair * 256 + rb + k;
                if (rb + k >= r1 || t >= p.T || !lanes_d) continue;
                float mx = ml[k][0].x;
#pragma unroll
                for (int sp = 1; sp < kMaxSplits; ++sp) mx = fmaxf(mx, ml[k][sp].x);
                float lw = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int sp = 0; sp < kMaxSplits; ++sp) {
                    const float w = sp < p.splits ? ex2_approx(ml[k][sp].x - mx) : 0.f;
                    lw = fmaf(w, ml[k][sp].y, lw);
                    acc.x = fmaf(w, o[k][sp].x, acc.x);
                    acc.y = fmaf(w, o[k][sp].y, acc.y);
                    acc.z = fmaf(w, o[k][sp].z, acc.z);
                    acc.w = fmaf(w, o[k][sp].w, acc.w);
                }
                const float f = 256.f / lw;   // V was widened as V * 2^-8
                *reinterpret_cast<float4*>(p.out + ((size_t)t * p.H + h) * D + 4 * lane) =
                    make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
            }
        }
        // no CTA leaves while another may still read its shared memory
        cluster_sync_all();
        return;
    }
    // partial of this split: O * 2^8 (unnormalised) and (M, l) per row.  With a
    // cooperative launch this split merges rows [own0, own1) itself and reads its
    // own share of them from shared memory, so only the other rows go out.
    const int own0 = p.coop ? split * rows / p.splits : 0;
    const int own1 = p.coop ? (split + 1) * rows / p.splits : 0;
    for (int rr = warp; rr < rows; rr += kAttendThreads / 32) {
        const int t = pair * 256 + rr;
        if (t >= p.T || (rr >= own0 && rr < own1)) continue;
        const size_t pr = ((size_t)split * p.H + h) * p.Tstride + t;
        if (lanes_d) {
            const float4 o = *reinterpret_cast<const float4*>(sO + (size_t)rr * kORow + 4 * lane);
            *reinterpret_cast<float4*>(p.part_o + pr * D + 4 * lane) =
                make_float4(o.x * 256.f, o.y * 256.f, o.z * 256.f, o.w * 256.f);
        }
        if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + pr * 2) = sML[rr];
    }
    // Split merge.  Every CTA counts itself in, aborted or not.  Cooperative launch
    // (all CTAs resident at once): the splits of a (head, pair) wait for each
    // other (bounded) and each merges its share of the rows; a second counter
    // tells the last one out to reset both.  Otherwise the last split to arrive
    // merges all rows.  Either way one warp per row, four rows per warp at a
    // time with all their loads in flight.
    __threadfence();
    __syncthreads();
    const size_t unit = (size_t)h * (p.Tstride / 256) + pair;
    int* counter = p.counters + unit;
    int* done = p.counters + (size_t)p.H * (p.Tstride / 256) + unit;
    int r0 = 0, r1 = rows;
    if (p.coop) {
        // own0 and own1 are this split's share of the rows
        if (tid == 0) {
            atomicAdd(counter, 1);
            const uint64_t t0 = globaltimer_ns();
            int ok = 1;
            while (atomicAdd(counter, 0) < p.splits) {
                if ((long long)(globaltimer_ns() - t0) > p.timeout_ns) {
                    ok = 0;
                    if (atomicCAS(p.err, 0, KVRING_ETIMEOUT) == 0) {
                        p.err[1] = kKernelAttend;
                        p.err[2] = kWaitMerge;
                        p.err[3] = (int)blockIdx.x;
                    }
                    break;
                }
            }
            *sLast = ok;
        }
        __syncthreads();
        r0 = own0;
        r1 = own1;
        if (!*sLast) r1 = r0;   // gave up: merge nothing
        __threadfence();
    } else {
        if (tid == 0) *sLast = atomicAdd(counter, 1) == p.splits - 1;
        __syncthreads();
        if (!*sLast) return;
        __threadfence();
    }
    for (int rb = r0 + warp * kRowsAtOnce; rb < r1; rb += kRowsAtOnce * (kAttendThreads / 32)) {
        float2 ml[kRowsAtOnce][kMaxSplits];
        float4 o[kRowsAtOnce][kMaxSplits];
#pragma unroll
        for (int k = 0; k < kRowsAtOnce; ++k) {
            const int t = pair * 256 + rb + k;
            const bool mine = rb + k < r1 && t < p.T;
#pragma unroll
            for (int sp = 0; sp < kMaxSplits; ++sp) {
                ml[k][sp] = make_float2(-INFINITY, 0.f);
                o[k][sp] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sp < p.splits && mine) {
                    if (sp == split) {   // this split's own rows are still in its shared memory
                        ml[k][sp] = sML[rb + k];
                        if (lanes_d) {
                            const float4 v = *reinterpret_cast<const float4*>(sO + (size_t)(rb + k) * kORow + 4 * lane);
                            o[k][sp] = make_float4(v.x * 256.f, v.y * 256.f, v.z * 256.f, v.w * 256.f);
                        }
                    } else {
                        const size_t pr = ((size_t)sp * p.H + h) * p.Tstride + t;
                        ml[k][sp] = __ldcg(reinterpret_cast<const float2*>(p.part_ml + pr * 2));
                        if (lanes_d) o[k][sp] = __ldcg(reinterpret_cast<const float4*>(p.part_o + pr * D + 4 * lane));
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRowsAtOnce; ++k) {
            const int t = pair * 256 + rb + k;
            if (rb + k >= r1 || t >= p.T || !lanes_d) continue;
            float mx = ml[k][0].x;
#pragma unroll
            for (int sp = 1; sp < kMaxSplits; ++sp) mx = fmaxf(mx, ml[k][sp].x);
            float lw = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int sp = 0; sp < kMaxSplits; ++sp) {
                const float w = sp < p.splits ? ex2_approx(ml[k][sp].x - mx) : 0.f;
                lw = fmaf(w, ml[k][sp].y, lw);
                acc.x = fmaf(w, o[k][sp].x, acc.x);
                acc.y = fmaf(w, o[k][sp].y, acc.y);
                acc.z = fmaf(w, o[k][sp].z, acc.z);
                acc.w = fmaf(w, o[k][sp].w, acc.w);
            }
            const float inv = 1.f / lw;
            *reinterpret_cast<float4*>(p.out + ((size_t)t * p.H + h) * D + 4 * lane) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
    }
    if (p.coop) {
        // the last split out resets both counters (every split has passed its wait)
        __syncthreads();
        if (tid == 0 && atomicAdd(done, 1) == p.splits - 1) {
            *counter = 0;
            *done = 0;
        }
    } else if (tid == 0) {
        *counter = 0;
    }
}

// Launched with programmatic stream serialisation: its CTAs may start while the
// Q prep grid before it is still running; they wait for it (griddepcontrol.wait)
// before reading Q.  Their first K/V loads come before that wait: Q prep lets
// this grid start only after its own wait, so whatever wrote the ring before Q
// prep has finished by then.  The kernel's shared-memory attribute is set once
// per device by attend_max_clusters (kvring_create asks it for the ring's d, the
// allocation-free entry point for both), so a launch makes no other CUDA call
// and can be captured into a graph.
cudaError_t launch_attend(const AttendParams& p, const AttendMaps& maps, cudaStream_t s) {
    const int grid = p.H * p.npairs * p.splits;
    const int smem = p.d == 128 ? (int)AttendSmem<128>::kAlloc : (int)AttendSmem<64>::kAlloc;
    void (*kern)(AttendParams, AttendMaps) = p.d == 128 ? attend_kernel<128> : attend_kernel<64>;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kAttendThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;   // the splits of a (head, pair) wait for each other
    attr[1].val.cooperative = p.coop ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (p.cluster) {   // consecutive CTAs are the splits of one (head, pair)
        attr[2].id = cudaLaunchAttributeClusterDimension;
        attr[2].val.clusterDim.x = (unsigned)p.splits;
        attr[2].val.clusterDim.y = 1;
        attr[2].val.clusterDim.z = 1;
        cfg.numAttrs = 3;
    }
    return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

// Also sets the kernel's dynamic shared-memory attribute on the current device,
// which every launch needs.
int attend_max_clusters(int d, int splits) {
    const int smem = d == 128 ? (int)AttendSmem<128>::kAlloc : (int)AttendSmem<64>::kAlloc;
    void (*kern)(AttendParams, AttendMaps) = d == 128 ? attend_kernel<128> : attend_kernel<64>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)splits, 1, 1);
    cfg.blockDim = dim3(kAttendThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace kvring_impl
