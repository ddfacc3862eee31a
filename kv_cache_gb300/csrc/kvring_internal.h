// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda.h>
#include <stdint.h>

#include <string>

#include "../../include/kvring.h"

namespace kvring_impl {

constexpr int kTile = 128;          // slots per KV tile, query rows per Q tile
constexpr float kE4M3Max = 448.0f;

// Device error word: [0] = status (0 or KVRING_ETIMEOUT), [1] = kernel id,
// [2] = wait site, [3] = block index that gave up.
enum KernelId : int { kKernelAttend = 1, kKernelWrite = 2 };

// ---------------------------------------------------------------- write (K1)
struct WriteParams {
    CUtensorMap kmap;         // the chunk's K, 3-D {d, H, T} bf16 (as u16), box {d, 1, 16}
    CUtensorMap vmap;         // the chunk's V, the same
    CUtensorMap ropemap;      // the RoPE table, 2-D {d (u32: d/2 cos-sin pairs), max_position}, box {d, 16}
    const uint16_t* k;        // bf16 [T][H][d]
    const uint16_t* v;        // bf16 [T][H][d]
    uint8_t* k8;              // this layer's K ring  [H][Rpad][d]
    uint8_t* vt8;             // this layer's V ring  [H][d][Rpad] (slot-contiguous)
    float* kamax;             // [H][Rpad]
    float* vamax;             // [H][Rpad]
    const float2* rope;       // [max_position][d/2] (cos, sin)
    int64_t head;             // first slot of the chunk
    int64_t pos0;             // position of token 0
    int T, H, d, R, Rpad;
    int groups;               // 16-slot groups touched by the chunk
    int group0;               // first group in cyclic order
    int ngroups_ring;         // ceil(R / 16)
    int amax_tokens_per_block;
    int amax_blocks;          // ceil(T / amax_tokens_per_block)
    float* part;              // per-block amax partials [K|V][amax_blocks][H] (ring scratch)
    int* err;                 // the ring's device error word
    long long timeout_ns;     // bound of each device wait
    int skip_group;           // testing aid: the rows of this ring group are not loaded (-1 = off)
};
cudaError_t write_setup();                                        // function attributes, once per device
cudaError_t launch_write(const WriteParams& p, cudaStream_t s);   // one launch (clusters)
// Tensor maps of a write: the chunk's K and V (per call) and the RoPE table (per ring).
int write_input_maps(WriteParams& p);
int write_rope_map(CUtensorMap* map, const float2* rope, int64_t max_position, int d);
cudaError_t launch_write_amax(const WriteParams& p, cudaStream_t s);   // chunk amax partials (naive scheme)
int write_amax_tokens_per_block(int H, int d);

// ---------------------------------------------------------------- naive upkeep (comparison)
struct NaiveAppendParams {
    const uint16_t* k;        // new chunk bf16 [T][H][d]
    const uint16_t* v;
    const uint16_t* kw_src;   // window before the call, bf16 [H][Rpad][d], logical row order
    const uint16_t* vw_src;
    uint16_t* kw_dst;         // window after the call (the other buffer, or the same for a rewrite)
    uint16_t* vw_dst;
    const float* ka_src;      // chunk amax of each window row [H][Rpad]
    const float* va_src;
    float* ka_dst;
    float* va_dst;
    const float* part;        // amax partials of the chunk [K|V][amax_blocks][H]
    int amax_blocks;
    int T, H, d, Rpad;
    int keep;                 // rows kept: dst row r < keep is src row r + drop
    int drop;                 // oldest rows dropped
    int row_begin;            // first dst row written (rows below it are already in place)
};
cudaError_t launch_naive_append(const NaiveAppendParams& p, cudaStream_t s);

struct NaiveRefreshParams {
    const uint16_t* kw;       // window bf16 [H][Rpad][d]
    const uint16_t* vw;
    const float* ka;          // chunk amax of each row [H][Rpad]
    const float* va;
    uint8_t* k8;              // this layer's FP8 cache, as for the write-time ring
    uint8_t* vt8;
    float* kamax;
    float* vamax;
    const float2* rope;       // [max_position][d/2]
    int64_t pos0;             // position of row 0
    int count, H, d, Rpad;
};
cudaError_t launch_naive_refresh(const NaiveRefreshParams& p, cudaStream_t s);

// ---------------------------------------------------------------- rebase (K2)
struct RebaseParams {
    uint8_t* k8;              // all layers [L][H][Rpad][d]
    const float* kamax;       // all layers [L][H][Rpad]
    const float2* rope;       // [max_position][d/2]
    int L, H, d, Rpad;
    int pairs;                      // leading pairs of a row that turn (d/2; the time band for 3-D RoPE)
    int delta[KVRING_MAX_LAYERS];   // per layer; 0 = skip
    int count[KVRING_MAX_LAYERS];   // valid slots per layer
};
cudaError_t launch_rebase(const RebaseParams& p, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- Q prep (K3)
struct QPrepParams {
    const uint16_t* q;        // bf16 [T][H][d]
    uint8_t* q8;              // [H][Tpad][d]
    float* qamax;             // [H][Tpad]
    const float2* rope;
    int64_t pos0;
    int T, Tpad, H, d;
    int Tstride;              // row stride of q8 in rows (= Tpad_max)
};
cudaError_t launch_qprep(const QPrepParams& p, cudaStream_t s);

// ---------------------------------------------------------------- attention (K4)
struct AttendParams {
    const float* kamax;       // this layer [H][Rpad]
    const float* vamax;       // this layer [H][Rpad]
    const float* qamax;       // [H][Tstride]
    float* out;               // fp32 [T][H][d]
    float* part_o;            // fp32 [splits][H][Tstride][d]   (splits > 1)
    float* part_ml;           // fp32 [splits][H][Tstride][2]   (splits > 1)
    int* counters;            // [2][H][Tstride/256], zero between calls (splits > 1)
    int* err;                 // device error word
    int T, H, d, Rpad, Tstride;
    int count;                // valid slots
    int layer;
    int npairs;               // ceil(T / 256): pairs of 128-row query tiles
    int splits;               // KV splits per (head, query pair)
    int tiles_per_split;
    int ntiles;               // ceil(count / 128)
    float log2e_rsqrt_d;      // log2(e) / sqrt(d)
    long long timeout_ns;
    int skip_tile;            // testing aid: K/V load of this tile is not issued (-1 = off)
    int coop;                 // launched cooperatively: the splits of a (head, pair) merge together
    int cluster;              // the splits of a (head, pair) are one thread-block cluster and merge
                              // through distributed shared memory (no partials in global memory)
};
struct AttendMaps {
    CUtensorMap q8;           // 3-D {d, Tstride, H}
    CUtensorMap k8;           // 3-D {d, Rpad, L*H}
    CUtensorMap vt8;          // 3-D {Rpad, d, L*H}
};
cudaError_t launch_attend(const AttendParams& p, const AttendMaps& maps, cudaStream_t s);
// How many clusters of `splits` attention CTAs (head dim d) the device holds at once (0 on error).
int attend_max_clusters(int d, int splits);

size_t attend_smem_bytes(int d);

// Shared by the host translation units.
void set_thread_error(const std::string& msg);
// Tiled tensor map (no swizzle unless given, 256-byte L2 promotion, zeros out of
// bounds); KVRING_OK or KVRING_ECUDA.  strides: rank - 1 byte strides.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz);
int encode_u8_map(CUtensorMap* map, void* base, const cuuint64_t dims[3], const cuuint64_t strides[2],
                  const cuuint32_t box[3], CUtensorMapSwizzle swz);

}  // namespace kvring_impl
