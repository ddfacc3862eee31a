/*
 * kvring.h -- C ABI of the GB300 write-time KV cache for streaming video DiT attention.
 *
 * The operations follow three public reports of Runway's real-time "Characters"
 * serving work:
 *   [ai.info]     "Characters funziona in tempo reale su quattro H100, afferma Runway",
 *                 sections "La gestione della cache spostata al momento della scrittura"
 *                 and "Latenza dei turni e altre configurazioni GPU";
 *   [neurocartel] "Runway Characters realtime on 4 H100" (neurocartel.com),
 *                 section "Кэш: 240 attention calls и работа на запись";
 *   [wechild]     wechild.cn news item on Runway's real-time Characters inference
 *                 paper (untitled), paragraphs 6-8.
 * The pages give no API; the calls below follow their statement of the problem:
 * write once per chunk, read many times, rebase once per position reset.
 *
 * Conventions shared by every call
 *   - Return value: KVRING_OK (0) or a negative KVRING_E* code.  Nothing aborts,
 *     throws or exits across this ABI.  A call that fails a precondition leaves
 *     the ring unchanged; the message is available from kvring_last_error().
 *   - Device pointers are raw CUDA device addresses of the current device;
 *     `cuda_stream` is a cudaStream_t (NULL = legacy default stream).
 *   - Hot calls (write, attend, rebase) only enqueue work on the stream: no host
 *     synchronisation.  The caller keeps its input/output buffers alive until the
 *     stream reaches the call.  All calls on one ring must be ordered on a single
 *     stream by the caller (the ring's scratch buffers are shared between calls).
 *   - The ring owns every device buffer it allocates (FP8 K and V rings, per-slot
 *     chunk amax, RoPE table, Q scratch, split partials, error word).  The caller
 *     owns every buffer it passes in.
 *   - Layouts: token-major bf16 [n][H][d] for K, V, Q inputs; fp32 [n][H][d] for
 *     the attention output.  All element counts are in elements, not bytes.
 */
#ifndef KVRING_H
#define KVRING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------- */
#define KVRING_OK        0
#define KVRING_EINVAL   (-1)  /* an argument is out of range or a pointer is NULL          */
#define KVRING_ENOMEM   (-2)  /* a host or device allocation failed                          */
#define KVRING_ECUDA    (-3)  /* a CUDA runtime/driver call failed (message has the reason)  */
#define KVRING_ESTATE   (-4)  /* not valid now: attend before any write, n_q differs from the
                                 last write, or positions would pass max_position (rebase)  */
#define KVRING_ETIMEOUT (-5)  /* a bounded device-side wait ran out (see kvring_check_device) */
#define KVRING_ENODEV   (-6)  /* no sm_103 device is current                                 */

/* ---- configuration flags ----------------------------------------------------- */
/* Bookkeeping only: no device memory, no CUDA calls, data pointers may be NULL.
 * write/rebase update the host state exactly as a device ring would; attend and
 * snapshot return KVRING_EINVAL.  Used to validate schedules on hosts without a GPU. */
#define KVRING_FLAG_HOST_ONLY 0x1u
/* The naive cache upkeep the pages replaced, kept as a measured comparison
 * ([wechild] paragraph 7; [ai.info] "La gestione della cache...": before the
 * change, cache upkeep took 69.7 ms of a 239.2 ms step).  Each layer holds its
 * window as un-rotated bf16 K and V in logical order (oldest first) with each
 * row's chunk amax.  kvring_write appends the chunk and drops the oldest rows
 * by copying the window; a rewrite replaces the newest rows; kvring_rebase only
 * lowers the positions.  kvring_naive_refresh re-applies RoPE to the whole window
 * at its current positions and re-quantises K and V into the layer's FP8 cache
 * (row r -> slot r), the upkeep the naive scheme repeats before every attention
 * call; kvring_attend reads that cache.  Rows are never rotated twice, so the
 * cache equals a fresh rotation at the current positions.  Uses 4 bytes per
 * element more device memory than a write-time ring (two bf16 window copies). */
#define KVRING_FLAG_NAIVE_UPKEEP 0x2u
/* 3-D (time, height, width) video RoPE.  The pages do not give the layout; the
 * plain reading for a video token grid: a token's running index p (the position
 * the ring counts) is frame * S + s with S = frame_tokens tokens per frame and
 * frame_width tokens per row, so its coordinates are t = p / S,
 * h = (p % S) / frame_width, w = (p % S) % frame_width.  Pairs [0, pt) rotate by
 * t, the next ph pairs by h and the remaining pw = d/2 - pt - ph by w, each band
 * with its own frequencies theta^(-2k/d_band), d_band = 2 x its pairs.  Every
 * write is a whole number of frames (n_tokens % S == 0) and capacity % S == 0,
 * so a position reset moves whole frames: it turns only the time band, and
 * kvring_rebase reads and writes only the 16-byte pieces of K that hold time
 * pairs (ceil(pt / 8) of the d/16 pieces per row); every other pair keeps its
 * codes exactly. */
#define KVRING_FLAG_ROPE_3D 0x4u

#define KVRING_MAX_LAYERS 256

typedef struct kvring kvring_t;       /* opaque */

typedef struct {
    int32_t  num_layers;             /* transformer blocks, each with its own ring: 1..256   */
    int32_t  num_heads;              /* H: 1..256                                            */
    int32_t  head_dim;               /* d: 64 or 128                                         */
    int32_t  capacity;               /* R: slots per ring, 1..1048576                        */
    int32_t  max_tokens_per_write;   /* T_max: 1..min(capacity, 2048)                        */
    int32_t  max_position;           /* positions must stay below this; 0 -> 65536.  Sets the
                                        size of the RoPE table (max_position x d/2 x 8 bytes) */
    float    rope_theta;             /* RoPE base; 0 -> 10000                                */
    uint32_t flags;                  /* KVRING_FLAG_*                                        */
    /* KVRING_FLAG_ROPE_3D only (ignored otherwise): */
    int32_t  frame_tokens;           /* S: tokens per frame, >= 1, divides capacity          */
    int32_t  frame_width;            /* tokens per row of a frame, >= 1, divides S           */
    int32_t  rope_pairs_t;           /* pt: pairs of the time band; 0 -> d/2 - 2*floor(d/6)  */
    int32_t  rope_pairs_h;           /* ph: pairs of the height band; 0 -> floor(d/6)        */
} kvring_config;

typedef struct {
    int64_t head;               /* next slot to write                                   */
    int64_t count;              /* valid slots: slots [0, count) hold data              */
    int64_t next_pos;           /* position of the next written token                   */
    int64_t writes;             /* chunks written to this layer (the next chunk's id)   */
    int64_t resets;             /* rebases applied (ring-wide)                          */
    int64_t last_write_pos;     /* position of the first token of the latest chunk      */
    int64_t last_write_tokens;  /* size of the latest chunk (0 before any write)        */
} kvring_state;

/* Create a ring set of cfg->num_layers rings.  Allocates all device memory on the
 * current device and builds the RoPE table on the host (angles p*w_i formed and
 * evaluated in float64, rounded once to float32; w_i = theta^(-2i/d)).
 * Slots start empty and zeroed.  *out receives the handle (NULL on failure).
 * Errors: EINVAL (bad config), ENODEV, ENOMEM, ECUDA. */
int kvring_create(const kvring_config* cfg, kvring_t** out);

/* Free every buffer the ring owns.  The caller makes sure no stream still uses it.
 * NULL is accepted and ignored. */
int kvring_destroy(kvring_t* ring);

/* Write one chunk of n_tokens new tokens into layer `layer`'s ring
 * ([ai.info] "La gestione della cache..."; [neurocartel] "Кэш...").
 *   k_bf16, v_bf16: device, bf16 [n_tokens][H][d], token-major, contiguous,
 *                   16-byte aligned (EINVAL otherwise).
 * One kernel launch: one cluster of 8 CTAs per (head, K|V), each CTA reading its
 * share of the chunk once into shared memory; the chunk amax is exchanged
 * between the CTAs of a cluster through distributed shared memory.
 * Token j goes to slot (head + j) mod R at position next_pos + j; the oldest slots
 * are overwritten, nothing is copied.  K is rotated by RoPE at its position and
 * both K and V are quantised to FP8 e4m3 with one scale per (head, chunk):
 * K amax = the largest RoPE-pair norm of the chunk, V amax = the largest |v|;
 * code = e4m3_rne_satfinite(x * (448/amax)).  The chunk's amax is stored with
 * each of its slots and never changes.
 * Then head += n (mod R), count = min(count + n, R), next_pos += n.
 * n_tokens == 0 is a no-op.  Errors: EINVAL (layer, pointers or their alignment, n_tokens >
 * max_tokens_per_write, or not a whole number of frames on a 3-D ring), ESTATE
 * (next_pos + n_tokens > max_position), ECUDA. */
int kvring_write(kvring_t* ring, int32_t layer, const void* k_bf16, const void* v_bf16,
                 int32_t n_tokens, void* cuda_stream);

/* Flags of kvring_write_ex. */
#define KVRING_WRITE_REWRITE 0x1u   /* replace the latest chunk instead of appending one */

/* kvring_write with flags.  flags == 0 is kvring_write.
 * KVRING_WRITE_REWRITE: the latest chunk of `layer` is written again with new K, V
 * and nothing advances.  A denoising model runs every block several times per
 * step ([ai.info] "La gestione della cache...": four passes through the 60
 * blocks, 240 attention calls per step), and the newest chunk's K and V are new
 * on each pass; the pages do not say how the cache takes them, and this call is
 * the plain reading: the same slots (head - n_tokens ... head - 1) mod R, the same
 * positions (last_write_pos + j, after any rebase since), the same chunk id, and
 * a new frozen scale per (head, chunk) from the new amax.  head, count,
 * next_pos and the write counter do not change; attend keeps reading the chunk
 * as the latest one.  Slots of older chunks are never touched.
 * Errors: as kvring_write, plus EINVAL (unknown flag bits) and ESTATE (rewrite
 * before any write to the layer, or n_tokens != the latest write's n_tokens;
 * n_tokens == 0 is a no-op only without the flag). */
int kvring_write_ex(kvring_t* ring, int32_t layer, const void* k_bf16, const void* v_bf16,
                    int32_t n_tokens, uint32_t flags, void* cuda_stream);

/* Attention of the latest chunk's queries over the finished FP8 cache of `layer`
 * ([wechild] paragraph 6; [ai.info] "Latenza dei turni...": FP8 attention that
 * accepts per-head scales).
 *   q_bf16:  device, bf16 [n_q][H][d]; query i sits at position last_write_pos + i.
 *   out_f32: device, fp32 [n_q][H][d].
 * Q is rotated at its positions and quantised to e4m3 per (token, head) row.
 * O = softmax(Q K^T / sqrt(d)) V over the valid slots, non-causal, every scale
 * applied per slot.  n_q must equal the latest write's n_tokens (0 is a no-op).
 * Errors: EINVAL, ESTATE (no write yet, n_q mismatch), ECUDA. */
int kvring_attend(kvring_t* ring, int32_t layer, const void* q_bf16, int32_t n_q,
                  float* out_f32, void* cuda_stream);

/* Naive per-call upkeep of one layer (rings created with KVRING_FLAG_NAIVE_UPKEEP):
 * rows [0, count) of the bf16 window are rotated by RoPE at positions
 * next_pos - count + r, quantised to e4m3 with their chunk scales (the same rules
 * as kvring_write) and stored in slots [0, count) of the layer's FP8 cache with
 * their chunk amax.  kvring_attend on a naive ring returns ESTATE unless the
 * layer was refreshed after its latest write, rewrite or rebase.
 * Errors: EINVAL (layer, or not a naive ring), ESTATE (no write yet), ECUDA. */
int kvring_naive_refresh(kvring_t* ring, int32_t layer, void* cuda_stream);

/* Position reset of every layer ([ai.info] "La gestione della cache...": positions
 * reset every 42 steps, one delta rotation of the cached window per reset).
 * For each layer delta = next_pos - count; every cached K is de-quantised,
 * rotated by -delta and re-quantised with its slot's frozen scale, in place;
 * V is untouched; positions drop by delta and next_pos = count.  Layers with
 * delta == 0 are skipped.  Errors: EINVAL, ECUDA. */
int kvring_rebase(kvring_t* ring, void* cuda_stream);

/* Host copy of one layer's bookkeeping (no device access).  Errors: EINVAL. */
int kvring_get_state(const kvring_t* ring, int32_t layer, kvring_state* out);

/* Synchronous copy of one layer's cache to caller-owned host buffers (tests, debug).
 *   host_k, host_v:         uint8 [H][R][d] e4m3 codes (either may be NULL)
 *   host_kamax, host_vamax: fp32  [H][R] chunk amax of each slot (either may be NULL)
 *   host_pos, host_chunk:   int32 [R] position / chunk id of each slot, -1 if empty
 * Enqueues the copies on cuda_stream and synchronises it.  Errors: EINVAL, ECUDA. */
int kvring_snapshot(const kvring_t* ring, int32_t layer, uint8_t* host_k, uint8_t* host_v,
                    float* host_kamax, float* host_vamax, int32_t* host_pos,
                    int32_t* host_chunk, void* cuda_stream);

/* Synchronous copy of the latest attention call's prepared queries (tests, debug):
 * the e4m3 codes of Q rotated at its positions, quantised per (token, head) row
 * with that row's own amax ([ai.info] "Latenza dei turni...": FP8 attention; the
 * query side is quantised the same way as the cache).
 *   host_q8:    uint8 [H][n_q][d] codes (may be NULL)
 *   host_qamax: fp32  [H][n_q] row amax, the largest |q| of the rotated row (may be NULL)
 * n_q is the latest kvring_attend's n_q.  Enqueues the copies on cuda_stream and
 * synchronises it.  Errors: EINVAL (NULL ring, host-only ring), ESTATE (no
 * attention call yet), ECUDA. */
int kvring_snapshot_q(const kvring_t* ring, uint8_t* host_q8, float* host_qamax, void* cuda_stream);

/* Synchronise cuda_stream and read the ring's device error word, which kernels set
 * when a bounded wait runs out.  Returns KVRING_OK or KVRING_ETIMEOUT (and clears
 * the word; the message says which kernel and wait).  Errors: EINVAL, ECUDA. */
int kvring_check_device(kvring_t* ring, void* cuda_stream);

/* Message of the last failed call on this ring (or of the last failed
 * kvring_create when ring is NULL).  Never NULL; valid until the next call. */
const char* kvring_last_error(const kvring_t* ring);

/* Number of kernels this ring has launched since it was created (every write,
 * attend and rebase adds the launches it enqueued).  Errors: EINVAL. */
int kvring_launch_count(const kvring_t* ring, uint64_t* out);

/* Testing aid for the bounded waits: make the next kvring_attend skip the K/V
 * load of tile `skip_tile` (-1 = off) and give each device wait timeout_ns
 * nanoseconds (0 = default of 2 s).  The skipped load makes its consumer's wait
 * run out; the kernel then records KVRING_ETIMEOUT, waits (bounded) for its own
 * copies in flight, frees its tensor memory and returns.  Errors: EINVAL. */
int kvring_debug_fault(kvring_t* ring, int32_t skip_tile, int64_t timeout_ns);

/* The same for the write kernel: the next kvring_write / kvring_write_ex (on a
 * ring without KVRING_FLAG_NAIVE_UPKEEP) leaves out the TMA copy of ring group
 * skip_group's rows (16 slots: skip_group * 16 ..) and gives each device wait
 * timeout_ns nanoseconds (0 = default of 2 s).  The CTA that waits for those
 * rows records KVRING_ETIMEOUT (kernel: write), still takes part in its
 * cluster's exchange, waits (bounded) for its other copies and returns without
 * storing; the chunk's codes are then unreliable until it is written again.
 * Errors: EINVAL. */
int kvring_debug_fault_write(kvring_t* ring, int32_t skip_group, int64_t timeout_ns);

/* Attention over a caller-held cache that allocates nothing.
 *
 * The pages have no counterpart to this call; it exists for callers that may
 * not allocate device memory (no cudaMalloc/cudaFree, no allocating library
 * routine) because their own arena or pool owns all of it, e.g. a serving
 * engine that places the FP8 cache in a slab it carved out itself.  It runs the
 * same Q preparation and FP8 attention as kvring_attend on one layer's cache,
 * given in these layouts (all device memory, caller-owned):
 *   k8:    e4m3 codes [H][slots_padded][d], slot-major rows, K already rotated
 *   vt8:   e4m3 codes [H][d][slots_padded], slot-contiguous rows
 *   kamax, vamax: fp32 [H][slots_padded], the chunk amax of each slot
 *          (scale = amax / 448, amax 0 meaning scale 1)
 *   rope:  fp32 (cos, sin) pairs [rope_rows][d/2]; entry [p][i] = fp32(cos(p * w_i)),
 *          fp32(sin(p * w_i)), angle and cosine in float64, w_i = theta^(-2i/d)
 *          (the table kvring_create builds).  The queries read rows q_pos0 ..
 *          q_pos0 + n_q - 1, so rope_rows >= q_pos0 + n_q (checked: EINVAL).
 *   q_bf16: [n_q][H][d]; query i sits at position q_pos0 + i
 *   out_f32: [n_q][H][d]
 * Slots [0, count) are attended; slots_padded is a multiple of 128 and the K
 * and V codes of slots [count, slots_padded) must be finite (zero will do): they
 * get weight exactly 0, but 0 times a NaN code is not 0.  k8, vt8, kamax,
 * vamax, q and out are 16-byte aligned.
 * err_word: 4 ints, zero before the call.  If a bounded device wait runs out the
 * kernel sets it to KVRING_ETIMEOUT (then kernel, wait site, block), but only
 * while word 0 is still zero: the call does not clear it, so it keeps the first
 * time-out of a series of calls until the caller zeroes it again.  NULL: the
 * library's own word is used, cleared on the stream at the start of every call,
 * and time-outs go unreported.
 *
 * Its only scratch is a fixed array inside the library (the e4m3 Q rows and
 * their amax): 16,384 rows of (head, query padded to 256), i.e. 2.06 MB that
 * every GPU loading the library holds until the process exits.  Larger calls
 * are rejected with KVRING_EINVAL.  The first call on a device looks up that
 * array's device address and how many attention clusters the device holds
 * (once per device); make that first call before any stream capture.  Every call shares the array and leaves its last contents
 * there; each call rewrites all of it that it reads, but calls that overlap on
 * the GPU (other streams, other threads) race and must be serialised by the
 * caller.  KV splits, when the call has them, merge as thread-block clusters
 * (no partials in memory), so it splits only where every cluster fits on the
 * device at once and may fill fewer SMs than kvring_attend.  Asynchronous on
 * cuda_stream.  Errors (message in kvring_last_error(NULL)): EINVAL, ENODEV,
 * ECUDA. */
int kvring_attend_noalloc(const void* k8, const void* vt8, const float* kamax, const float* vamax,
                          const float* rope, int64_t rope_rows, int64_t q_pos0, const void* q_bf16, int32_t n_q,
                          int32_t num_heads, int32_t head_dim, int32_t slots_padded, int32_t count,
                          float* out_f32, int* err_word, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* KVRING_H */
