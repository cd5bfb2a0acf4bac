/*
 * whead.h — C ABI of the walk-resident serial draft head for GB300 (sm_103a).
 *
 * The operation ("Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding",
 * abstract; Figs. 1, 2, 7, 8): a parallel block drafter has produced base logits for gamma positions;
 * a light serial head then walks those positions one by one. Step t projects a small state u_t (rank r)
 * through one immutable V x r matrix W, adds the base logits, picks one token over all V rows (greedy,
 * or Gumbel-max sampling at temperature T), and advances the state from the picked token:
 *   Markov head:    u_{t+1} = E[x_t]
 *   recurrent head: h_{t+1} = tanh(A h_t + E[x_t] + c), u_t = h_t
 * The state is rounded to bf16 before the projection; the projection accumulates in fp32; z = p + base
 * is formed in fp32 and rounded once when it is emitted; ties go to the smallest row index. The noise
 * for T > 0 is Philox4x32-10 keyed on (seed lo, seed hi) with counter (v/4, t0 + t, b, 0), word v%4,
 * U = ((w >> 9) + 0.5) * 2^-23, g = -log(-log U), key = z / T + g.
 *
 * Execution: one persistent cooperative kernel per walk. Each CTA keeps its shard of W on chip (shared
 * memory, tensor memory and registers) for the whole walk and exchanges only packed {key, row} words and
 * the compact state between steps (Fig. 1; Fig. 8).
 *
 * Conventions for every call below:
 *  - Pointers named W, E, A, c, base, u0/s0 and out_* are DEVICE pointers unless the name says host.
 *  - W, E (and A, c) are borrowed for the lifetime of the handle and must not change (W is immutable
 *    for the whole walk). Call inputs and outputs are borrowed for the call; the caller allocates them.
 *  - The handle owns only its scratch (exchange slots, counters, status word, staging buffers).
 *  - Calls are asynchronous on the handle's stream unless stated otherwise. Calls on one handle must be
 *    ordered on that stream (they share the handle's scratch).
 *  - Return values: WHEAD_OK or a negative WHEAD_ERR_* code. A device-side failure (a wait that ran past
 *    its time limit) is reported by whead_status() and by the next call on the handle.
 */
#ifndef WHEAD_H_
#define WHEAD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WHEAD_OK 0
#define WHEAD_ERR_INVALID_ARG (-1)  /* a null pointer, a size out of range, a misaligned pointer */
#define WHEAD_ERR_UNSUPPORTED (-2)  /* shape outside what this build handles (see whead_create) */
#define WHEAD_ERR_CUDA (-3)         /* a CUDA runtime or driver call failed */
#define WHEAD_ERR_TIMEOUT (-4)      /* a device-side wait gave up after its time limit */
#define WHEAD_ERR_NO_COOP (-5)      /* the grid cannot be made co-resident (cooperative launch refused) */
#define WHEAD_ERR_INTERNAL (-6)     /* a device-side consistency check failed */

typedef enum { WHEAD_MARKOV = 0, WHEAD_RECURRENT = 1 } whead_kind;

/* Flags (whead_params.flags). */
#define WHEAD_FLAG_LOGITS_F32 (1u << 0)      /* out_logits holds fp32 z instead of bf16(z) */
#define WHEAD_FLAG_FIXED_LATENT (1u << 1)    /* measurement mode: never advance the state (Fig. 13b probe) */
#define WHEAD_FLAG_FORCE_STREAM (1u << 2)    /* measurement mode: keep no row of W on chip; every step re-reads all
                                                of W from L2/HBM (the fused but non-resident walk of Figs. 4, 11) */
#define WHEAD_FLAG_PLACEMENT_CAPS (1u << 3)  /* measurement mode (Fig. 12's placement sweep): cap_smem, cap_tmem and
                                                cap_rf bound the 16-row groups per CTA that shared memory, tensor
                                                memory and registers may hold; the rest are streamed. Without the
                                                flag the planner fills shared memory, then tensor memory, then
                                                registers, and the cap fields are ignored. */
#define WHEAD_FLAG_W_E4M3 (1u << 4)  /* E4M3 weights (the pages' Fig. 7 two-vector projection, with the 8-bit float
                                        format that GB300's tensor cores run fast): whead_create quantizes W into a
                                        handle-owned copy (whead_quantize_w_e4m3), and every step splits the state
                                        into two scaled E4M3 vectors whose projections are scaled and summed.
                                        Requires r = 128 or 256 and max_B <= 4; not with whead_walk_noalloc. */
#define WHEAD_FLAG_HOST_STAGE (1u << 5)  /* whead_walk_host copies base logits and u0 in and the tokens out through
                                           device buffers even where the GPU could reach the caller's memory */
#define WHEAD_FLAG_FAULT_SKIP_ARRIVAL (1u << 8) /* testing: CTA 0 never arrives at step 0's exchange, so
                                                   every other CTA's bounded wait runs out */

typedef struct {
  int32_t kind;        /* WHEAD_MARKOV or WHEAD_RECURRENT */
  int32_t r;           /* rank: 64, 128, 192 or 256 */
  int64_t V;           /* vocabulary rows: 1 <= V < 2^24 */
  const float* A;      /* recurrent only: r x r fp32 row-major, device */
  const float* c;      /* recurrent only: r fp32, device; NULL means zero */
  int32_t max_B;       /* largest batch a call will use: 1..16 */
  int32_t max_gamma;   /* largest number of steps a call will use: 1..64 */
  void* stream;        /* cudaStream_t for every call on this handle; NULL = legacy default stream */
  uint32_t flags;      /* WHEAD_FLAG_* */
  int32_t grid;        /* number of CTAs; 0 = chosen by the planner (at most one per SM) */
  uint32_t timeout_us; /* limit on every device-side wait; 0 = 1,000,000 us */
  int32_t cap_smem;    /* with WHEAD_FLAG_PLACEMENT_CAPS: most groups per CTA in shared memory (>= 0) */
  int32_t cap_tmem;    /* with WHEAD_FLAG_PLACEMENT_CAPS: most groups per CTA in tensor memory (>= 0) */
  int32_t cap_rf;      /* with WHEAD_FLAG_PLACEMENT_CAPS: most groups per CTA in registers (>= 0) */
  int64_t v_offset;    /* vocabulary sharding: global index of W's first row (a multiple of 16; 0 for a whole
                          vocabulary). Rows of W are rows v_offset .. v_offset + V - 1 of the vocabulary:
                          tokens, packed keys and the noise counters use global rows, and E must hold the
                          global rows (E is indexed by the winner). */
  int64_t e_rows;      /* rows of E (0 = v_offset + V); winners handed to whead_advance must be below it */
} whead_params;

/* Placement chosen for a batch size (whead_plan_info). Groups are 16 consecutive rows of W. */
typedef struct {
  int32_t grid;            /* CTAs (one per SM) */
  int32_t threads;         /* threads per CTA */
  int32_t groups_per_cta;  /* 16-row groups each CTA owns */
  int32_t smem_groups;     /* of which resident in shared memory */
  int32_t tmem_groups;     /* of which resident in tensor memory */
  int32_t rf_groups;       /* of which resident in registers */
  int32_t stream_groups;   /* of which re-read from L2/HBM every step */
  int32_t smem_bytes;      /* dynamic shared memory per CTA */
  int32_t tmem_cols;       /* tensor-memory columns allocated per CTA */
  int32_t sm_count;        /* SMs on the device */
} whead_plan;

typedef struct whead_s whead_t;

/*
 * Create a handle for one head (abstract: the serial head of a parallel drafter; Fig. 1: each SM keeps
 * a shard of W). Validates shapes, queries the device, plans the placement of W over shared memory,
 * tensor memory and registers for B <= 8 and B <= 16, builds the TMA descriptor of W and allocates the
 * scratch. W and E: V x r bf16 row-major device arrays, 16-byte aligned. Returns WHEAD_ERR_UNSUPPORTED if
 * r is not one of 64/128/192/256, if V >= 2^24, if the recurrent head is asked for without A, or if W
 * cannot be placed for max_B. On success *out owns the scratch; free it with whead_destroy.
 */
int whead_create(const void* W, const void* E, const whead_params* params, whead_t** out);

/*
 * One walk of gamma steps for B independent walks (abstract; Fig. 2; Fig. 8). base: B x gamma x V fp32;
 * u0: B x r fp32 (the state projected at step 0); T >= 0 (0 = greedy); seed keys the noise.
 * out_tokens: B x gamma int32. out_logits: NULL, or B x gamma x V bf16 (fp32 with WHEAD_FLAG_LOGITS_F32)
 * holding z before noise and temperature. Enqueued on the handle's stream.
 */
int whead_walk(whead_t* h, const float* base, const float* u0, int32_t B, int32_t gamma, float T,
               uint64_t seed, int32_t* out_tokens, void* out_logits);

/*
 * whead_walk with a resume offset: the walk starts at absolute step t0 (which keys the noise) from state
 * s0 (B x r fp32), and out_state (NULL, or B x gamma x r fp32) receives the state after each step's
 * advance. Re-running from any step t0 with the state reached there reproduces the remaining tokens,
 * logits and states bit for bit.
 */
int whead_walk_ex(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T,
                  uint64_t seed, int64_t t0, int32_t* out_tokens, void* out_logits, float* out_state);

/*
 * whead_walk_ex that also returns each step's winning packed key (out_keys: NULL, or B x gamma uint64,
 * device, 8-byte aligned): ord(key) << 32 | (2^32 - 1 - row), where key is the winner's selection key (z, or
 * z / T + Gumbel noise), ord maps fp32 to uint32 in order (negative values ~bits, others bits | 2^31, -0 as +0)
 * and row is the global row. The largest key over shards is the winner over the union of their rows, ties
 * going to the lowest row (Fig. 8's packed selection, taken across GPUs for a sharded vocabulary).
 */
int whead_walk_keys(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T,
                    uint64_t seed, int64_t t0, int32_t* out_tokens, uint64_t* out_keys, void* out_logits,
                    float* out_state);

/*
 * The state after one step for given winners (abstract: the state advance, done on the GPU): x (B int32,
 * global rows of E, device), s (B x r fp32, the state that step projected, device) -> s_next (B x r fp32,
 * device). Markov: s_next = E[x]; recurrent: tanh(A s + E[x] + c), in the walk kernel's order of operations.
 * Enqueued on the handle's stream. A winner outside E gives a zero state and the device status
 * WHEAD_ERR_INTERNAL (see whead_status). For a vocabulary sharded over GPUs, every rank advances with the
 * winner of the merged keys.
 */
int whead_advance(whead_t* h, const int32_t* x, const float* s, float* s_next, int32_t B);

/*
 * Synchronous walk on HOST buffers (same arguments and layouts as whead_walk; every pointer may be host
 * memory, pinned or not, and the caller keeps ownership). The base logits (B x gamma x V fp32, about
 * 9.7 MB for B = 1, gamma = 16, V = 151,936) are read by the walk where they lie whenever this GPU can
 * address that memory: host memory pinned by CUDA, or any host memory on systems whose GPU walks the
 * host's page tables (Grace with NVLink-C2C), as well as device or managed memory. Otherwise, or with
 * WHEAD_FLAG_HOST_STAGE, they are first copied to a handle-owned device buffer. u0 is copied to the device,
 * the walk runs on the handle's stream, the tokens (and logits, if requested) are copied back, and the call
 * waits for the stream. Returns WHEAD_OK, an argument or CUDA error, or the first device-side error of the
 * handle's stream (WHEAD_ERR_TIMEOUT, WHEAD_ERR_INTERNAL), which it then clears as whead_status does; the
 * outputs are undefined after a device-side error.
 */
int whead_walk_host(whead_t* h, const float* base_host, const float* u0_host, int32_t B, int32_t gamma,
                    float T, uint64_t seed, int32_t* out_tokens_host, void* out_logits_host);

/*
 * Profiling aid: phase stamps of every CTA for the following walks on this handle (NULL turns it off).
 * trace: device buffer of uint64, 8-byte aligned, of at least grid x S x 8 bytes with S = 4 + 8 * gamma
 * (grid from whead_plan_info); a walk that does not fit writes no stamps. Row c (S words) of CTA c holds
 * S/2 SM-clock stamps followed by the same S/2 stamps as global-timer nanoseconds: [0] kernel start,
 * [1] shard loaded, then for step t at 2 + 4t: step start, projection and local selection done, exchange
 * done (thread 0 saw every CTA's arrival), state advanced.
 */
int whead_set_trace(whead_t* h, void* trace, int64_t bytes);

/* Waits for the handle's stream and returns WHEAD_OK or the first device-side error (then clears it). */
int whead_status(whead_t* h);

/* The placement used for batch size B (1..max_B). */
int whead_plan_info(const whead_t* h, int32_t B, whead_plan* out);

/*
 * The placement whead_create would choose (Fig. 1: each SM keeps a shard of W; Fig. 12: its split over the
 * on-chip tiers), computed on the host alone: no device is queried or touched, so it also serves planning
 * and tests on machines without a GPU. Arguments as in whead_params (max_B, the batch size B in 1..max_B,
 * flags: only WHEAD_FLAG_W_E4M3 is read) plus the device's SM count and opt-in shared memory per block in
 * bytes. Fills *out (sm_count as given). work_lists, if not NULL, receives 12 rows of 33 uint32 words, one
 * row per warp: its number of groups, then up to 32 entries (bits 0..7 the CTA-local group, bits 8..9 its
 * tier: 0 shared memory, 1 tensor memory, 2 registers, 3 streamed; bits 16..25 its first tensor-memory
 * column). rf_warp_mask (nullable) receives the warps that keep a group in registers, ah_warp (nullable) the
 * warp that computes a recurrent head's slice of A h. Returns WHEAD_ERR_INVALID_ARG for bad arguments and
 * WHEAD_ERR_UNSUPPORTED when the shape is not supported or W cannot be placed.
 */
int whead_plan_query(int64_t V, int32_t r, int32_t kind, int32_t max_B, int32_t B, uint32_t flags, int32_t sm_count,
                     int32_t smem_optin, whead_plan* out, uint32_t* work_lists, uint32_t* rf_warp_mask,
                     int32_t* ah_warp);

/*
 * E4M3 weights: quantizes W (V x r bf16, device, 16-byte aligned) row by row into Wq (V x r E4M3 codes,
 * device, 16-byte aligned, caller-owned) and sw (V fp32 row scales, device): s = max_k |W[v,k]| / 448 (fp32),
 * inv = 1 / s (fp32, correctly rounded, formed once per row), Wq[v,k] = E4M3(W[v,k] * inv) rounded to nearest
 * even and saturated at +-448; a row whose largest magnitude is below 448 * FLT_MIN (inv would not be finite)
 * gets s = 0 and zero codes. Enqueued on `stream` (cudaStream_t, NULL = legacy default). r must be 128 or 256.
 * Returns WHEAD_ERR_INVALID_ARG for null or misaligned pointers, WHEAD_ERR_UNSUPPORTED for other shapes.
 */
int whead_quantize_w_e4m3(const void* W, int64_t V, int32_t r, void* Wq, float* sw, void* stream);

/* A static description of a return code. */
const char* whead_strerror(int code);

/* Frees the handle and its scratch. Waits for the handle's stream first. */
int whead_destroy(whead_t* h);

/*
 * Walk without any device allocation. The paper has no counterpart: this entry point exists for callers
 * that must not call cudaMalloc, such as serving engines that reserve all GPU memory up front in their own
 * pool (an extra cudaMalloc may fail or bypass the pool's accounting) and latency-critical loops where a
 * cudaMalloc/cudaFree would synchronize the device. It runs the same walk as whead_walk with no handle:
 * the placement and the TMA descriptor of W are built on the host for every call, and the walk's scratch
 * (exchange slots, arrival counter, A h slices, status word) lives in one file-scope device array of
 * WHEAD_NOALLOC_SCRATCH_BYTES that every GPU loading this library keeps until the process exits.
 *
 * Arguments: W, E and params as for whead_create (params->max_B, max_gamma and grid are ignored: the call
 * plans for its own B and gamma; params->stream is the stream used); base, u0, B, gamma, T, seed,
 * out_tokens and out_logits as for whead_walk. out_status: NULL, or a device int32 that receives the
 * call's device status (0, or WHEAD_ERR_TIMEOUT / WHEAD_ERR_INTERNAL) once the stream reaches the end of
 * the walk. With out_status NULL a device-side failure is not reported anywhere (the call has already
 * returned WHEAD_OK and the tokens are then undefined): pass a status word to learn of it. All pointers are
 * device pointers owned by the caller.
 *
 * Errors: WHEAD_ERR_INVALID_ARG / WHEAD_ERR_UNSUPPORTED as whead_create and whead_walk; a call whose
 * scratch would exceed WHEAD_NOALLOC_SCRATCH_BYTES is rejected with WHEAD_ERR_UNSUPPORTED: more than 16
 * walks or more than 64 steps. The grid is at most 256 CTAs (the array's slots per step); on a device with
 * more SMs the walk uses 256 of them. The measurement and staging flags (WHEAD_FLAG_FORCE_STREAM,
 * WHEAD_FLAG_PLACEMENT_CAPS, WHEAD_FLAG_HOST_STAGE) and WHEAD_FLAG_W_E4M3 need a handle and are rejected
 * with WHEAD_ERR_UNSUPPORTED.
 *
 * Every call shares the one array and clears what must start at zero (exchange slots, counter, status and,
 * for the recurrent head, the tagged A h slices) with cudaMemsetAsync on the call's stream. Calls whose walks overlap on the GPU (different streams, or several
 * host threads) race on the array and give wrong results: serialize them. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) and the device's limits; make that first call
 * before any stream capture.
 */
#define WHEAD_NOALLOC_SCRATCH_BYTES (192 * 1024)
int whead_walk_noalloc(const void* W, const void* E, const whead_params* params, const float* base,
                       const float* u0, int32_t B, int32_t gamma, float T, uint64_t seed, int32_t* out_tokens,
                       void* out_logits, int32_t* out_status);

#ifdef __cplusplus
}
#endif

#endif /* WHEAD_H_ */
