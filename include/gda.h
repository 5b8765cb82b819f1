/*
 * gda.h -- gated split-KV GQA decode attention on GB300 (sm_103a): the C ABI.
 *
 * One decode token per sequence attends, per query head, to the KV rows that a
 * CSR slot index names in a paged (page size 1) KV pool; the attention output is
 * then gated by the sigmoid of a second projection of the same shape:
 *
 *   out[b,h,:] = RNE_bf16( RNE_bf16(O[b,h,:]) * RNE_bf16(sigmoid(gate[b,h,:])) )
 *   O[b,h,:]   = softmax_j(scale * q[b,h,:] . K[slot_j, h/G, :]) V[slot_j, h/G, :]
 *   slot_j     = kv_indices[kv_indptr[b] + j],  0 <= j < kv_indptr[b+1]-kv_indptr[b]
 *
 * with G = Hq / Hkv consecutive query heads sharing one KV head (any G >= 1; the
 * kernels handle the query heads of a KV head in groups of up to 8: for G > 8 the
 * default kernel serves the groups in teams, every group of a team from one read of
 * the KV head's rows -- pairs for 2 or 4 groups, threes otherwise: one read for
 * G = 9 .. 24, two for 25 .. 48; an e4m3 cache's kernel takes pairs except for three
 * groups -- and the other kernels read the rows once per group).  Sources: FreeToken
 * PR #781 "Fuse the BF16 attention output sigmoid gate into the existing Triton
 * decode stage2" (Summary: split-KV stage 1, FP32 LSE merge in stage 2 with the
 * BF16 gate and an explicit round-to-nearest-even product fused into its epilogue;
 * Automatic dispatch: query [1,16,256], two KV heads, contiguous BF16 tensors, a
 * CSR index, default scale); cuDNN FE-OSS "Gated Attention Block (SM107)"
 * (Overview, stages (4) SDPA with GQA and (5) gate; Forward: the caller passes
 * one workspace, execute allocates nothing and reads nothing back).
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller (gda_decode_step_host
 *    also takes two HOST pointers, host_in and host_out).  The library never frees or
 *    retains them and never writes to an input.
 *  - Every tensor is contiguous and 16-byte aligned.  BF16 values are passed as
 *    their 16-bit patterns (gda_bf16).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and the call returns without waiting for it.  No call except
 *    gda_read_error (and gda_decode_step_host, whose job it is) reads anything back
 *    from the device.
 *  - The return value is GDA_OK (0) or a negative gda_status; on an error nothing
 *    has been enqueued.  Host-side checks (pointers, shapes, alignment, sizes) run
 *    before any CUDA call, so they work without a GPU.
 *  - Index contents are not validated on the host (that would need a read back):
 *    an index outside [0, num_slots) is undefined behaviour unless
 *    gda_args.check_indices is set.
 */
#ifndef GDA_H
#define GDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gda_bf16;                 /* bfloat16 bit pattern */
typedef struct CUstream_st* gda_stream_t;   /* the same type as cudaStream_t */

typedef enum gda_status {
    GDA_OK = 0,
    GDA_ERR_NULL = -1,          /* a required pointer is NULL */
    GDA_ERR_ALIGN = -2,         /* a pointer is not 16-byte aligned */
    GDA_ERR_SHAPE = -3,         /* B < 0, Hq < 1, Hkv < 1, Hq % Hkv != 0, num_slots < 0, n < 0 */
    GDA_ERR_UNSUPPORTED = -4,   /* a shape or option the built kernels do not serve (D != 256,
                                   an unknown variant): declined, never run slowly */
    GDA_ERR_SPLITS = -5,        /* num_splits > GDA_MAX_SPLITS */
    GDA_ERR_WORKSPACE = -6,     /* workspace NULL, misaligned or smaller than gda_workspace_bytes */
    GDA_ERR_CAPTURE = -7,       /* set-up needed while `stream` is capturing: the internal
                                   workspace must grow, or gda_prefill's first use on a device */
    GDA_ERR_CUDA = -8,          /* a CUDA runtime call or launch failed */
    GDA_ERR_DEVICE = -9,        /* gda_read_error: a kernel flagged an error (see the bits below) */
    GDA_ERR_ARG = -10           /* a scalar argument outside its domain (a non-finite descale) */
} gda_status;

#define GDA_MAX_SPLITS 256
/* Bits of the device error word (gda_read_error). */
#define GDA_DEVERR_INDEX 0x1u    /* an index outside [0, num_slots) (check_indices only) */
#define GDA_DEVERR_TIMEOUT 0x2u  /* a pipeline wait gave up (kernel bug guard; never expected) */

/* Stage-1 kernel variant (gda_args.variant). */
#define GDA_VARIANT_AUTO 0       /* the fastest built variant (GDA_VARIANT_MMA) */
#define GDA_VARIANT_MMA 1        /* K/V rows loaded straight into registers; QK and PV on
                                    mma.sync m16n8k16 bf16 tiles with FP32 accumulation */
#define GDA_VARIANT_SIMT 2       /* same loads; QK and PV as FP32 FMAs with warp-shuffle
                                    reductions */
#define GDA_VARIANT_TMA 3        /* K/V rows gathered into a shared-memory ring by 1-D bulk
                                    copies (TMA), then mma.sync tiles (comparison variant) */

/* Element type of the K and V pools (gda_args.kv_dtype). */
#define GDA_KV_BF16 0            /* bf16 values */
#define GDA_KV_E4M3 1            /* e4m3 codes (torch.float8_e4m3fn bytes) with per-tensor descales:
                                    K = k_descale * e4m3(code), V = v_descale * e4m3(code) */

/*
 * Full argument set of gda_decode_ex.
 *   q, gate     [B, Hq, D] bf16            query and gate of the decode token
 *   k_pool      [num_slots, Hkv, D] bf16   K rows, one token per slot (e4m3 bytes when
 *                                          kv_dtype == GDA_KV_E4M3)
 *   v_pool      [num_slots, Hkv, D] bf16   V rows (likewise)
 *   kv_indptr   [B + 1] int32              CSR row pointer, kv_indptr[0] == 0, non-decreasing
 *   kv_indices  [kv_indptr[B]] int32       slot of each position, in position order
 *   out         [B, Hq, D] bf16            result (may not alias an input)
 *   lse         [B, Hq] float or NULL      natural-log log-sum-exp of the scaled scores
 *                                          (-inf for a zero-length sequence)
 *   num_slots   rows in the pools (used only by check_indices)
 *   scale       score scale (1/sqrt(D) is the pages' default)
 *   num_splits  > 0: every sequence is cut into exactly num_splits contiguous KV
 *               splits (split s covers positions [s*c, min(L, (s+1)*c)), c = ceil(L/S));
 *               <= 0: automatic -- the kernel cuts the concatenated KV stream of the
 *               whole batch into equal chunks, one per resident CTA, from kv_indptr
 *               on the device (no read back), so ragged batches stay balanced.
 *   fuse_gate   1: out is the gated result.  0: out = RNE_bf16(O) without the gate (the
 *               first half of the unfused path; gda_gate is the second).
 *   check_indices 1: every index is checked on the device; a bad row is read as zeros and
 *               GDA_DEVERR_INDEX is set in the workspace's error word.
 *   variant     GDA_VARIANT_* (stage-1 arithmetic).
 *   min_chunk   automatic mode: smallest chunk in tokens per CTA (0: built-in default).
 *   window      > 0: sliding window -- sequence b attends only to its last `window`
 *               positions, kv_indices[kv_indptr[b+1] - min(L, window) .. kv_indptr[b+1]);
 *               0: all positions.  With num_splits <= 0 the split count is then chosen
 *               on the host (equal splits of the window).
 *   sinks       [Hq] float sink logits or NULL: attention sinks, one logit per query head
 *               that joins the softmax denominator with a zero value row,
 *               O = sum_j e^{s_j} V_j / (e^{sink_h} + sum_j e^{s_j}); lse includes it.
 *   kv_dtype    GDA_KV_BF16 or GDA_KV_E4M3 (an FP8 KV cache, cuDNN FE-OSS "Gated Attention
 *               Block (SM107)", API, QuantSpec: static per-tensor scales, e4m3 codes).
 *               E4M3 is served by GDA_VARIANT_AUTO / GDA_VARIANT_MMA only.
 *   k_descale, v_descale  per-tensor factors of an e4m3 cache (finite; else GDA_ERR_ARG);
 *               not used for bf16 pools.
 *   max_len     0, or an upper bound on every sequence's KV length that the caller knows
 *               on the host (a scheduler's batch maximum).  With a bound of at most
 *               1024, automatic splits (num_splits <= 0), GDA_VARIANT_AUTO, bf16 or e4m3
 *               pools, no check_indices, Hq / Hkv <= 8, and few enough (sequence, KV head) pairs
 *               (gda_small_path_cluster), the call runs as ONE kernel: a thread-block
 *               cluster of 8, 4, 2 or 1 CTAs per (sequence, KV head) (the most that fit in
 *               one wave, at most 128 positions per CTA) that merges its partial
 *               softmax states in distributed shared
 *               memory and applies the gate, with no workspace traffic.  The result
 *               is the same function within the tolerance of the split path.  A bound
 *               below an actual length still gives the right result, only slower.
 *   total_len   0, or the batch's exact number of KV positions (kv_indptr[B]) known on
 *               the host.  With max_len > 0 too, automatic splits and no window, the
 *               split count is chosen on the host (gda_auto_splits with lmax = max_len)
 *               and uniform splits launch as explicit ones: no scan of kv_indptr on the
 *               device and no idle CTAs.  A wrong value changes only the speed.
 * (FreeToken PR #781, Automatic dispatch and Correctness: window, sinks, custom scale
 * and non-power-of-two GQA groups are the cases of the general path.)
 */
typedef struct gda_args {
    const gda_bf16* q;
    const gda_bf16* gate;
    const void* k_pool;
    const void* v_pool;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    gda_bf16* out;
    float* lse;
    int64_t num_slots;
    int B, Hq, Hkv, D;
    float scale;
    int num_splits;
    int fuse_gate;
    int check_indices;
    int variant;
    int min_chunk;
    int window;
    const float* sinks;
    int kv_dtype;
    float k_descale;
    float v_descale;
    int max_len;
    int64_t total_len;
} gda_args;

/* Bytes of workspace gda_decode_ex needs for these sizes (FreeToken PR #781 Summary:
 * stage 1 writes per-split partial O and LSE that stage 2 merges).  The workspace
 * holds a 256-byte header (error word, plan), then FP32 partials
 * [pieces][8][D] and partial LSE [pieces][8].  Returns 0 for invalid sizes.  The
 * size for num_splits <= 0 also covers every call with a window. */
size_t gda_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits);

/* Zero the workspace header (error word) on `stream`.  Call once after allocating
 * a workspace for gda_decode_ex; partial buffers need no initialisation. */
int gda_workspace_init(void* workspace, size_t workspace_bytes, gda_stream_t stream);

/* Gated GQA decode attention with library-owned workspace (FreeToken PR #781,
 * Summary and Automatic dispatch).  Two kernels are enqueued: stage 1 (split
 * partial softmax(q K^T scale) V with running max and LSE) and stage 2 (FP32 LSE
 * merge and the BF16 gate epilogue), the second with programmatic dependent launch.
 * The internal workspace is one per device, shared by every stream: calls that may
 * overlap on different streams must use gda_decode_ex with separate workspaces.
 * It grows with cudaMalloc when needed (to at least twice its size, with a device
 * synchronisation); growth is refused with GDA_ERR_CAPTURE while `stream` is
 * capturing (call gda_reserve before capturing a graph).  A growth never frees the
 * buffer it replaces: a graph captured earlier keeps reading and writing that buffer
 * on replay, so it stays valid after later, larger calls.  Replaced buffers stay
 * allocated until the process exits (together less than the current one). */
int gda_decode(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k_pool,
               const gda_bf16* v_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
               gda_bf16* out, int B, int Hq, int Hkv, int D, float scale, int num_splits,
               gda_stream_t stream);

/* As gda_decode with the full argument set and a caller-owned workspace of at least
 * gda_workspace_bytes(B, Hq, Hkv, D, num_splits) bytes (256-byte aligned).
 * Allocates nothing and reads nothing back (cuDNN FE-OSS "Gated Attention Block
 * (SM107)", Forward: execute() allocates nothing), so it can be graph-captured. */
int gda_decode_ex(const gda_args* args, void* workspace, size_t workspace_bytes,
                  gda_stream_t stream);

/* As gda_decode over an FP8 KV cache: k_pool and v_pool hold e4m3 codes
 * ([num_slots, Hkv, D] bytes, 16-byte aligned) whose values are k_descale * e4m3(c)
 * and v_descale * e4m3(c) (cuDNN FE-OSS "Gated Attention Block (SM107)", API,
 * QuantSpec: static per-tensor scales; e4m3 as torch.float8_e4m3fn).  q and gate stay
 * bf16, the output and its rounding are those of gda_decode.  Same library-owned
 * workspace as gda_decode.  Non-finite descales: GDA_ERR_ARG. */
int gda_decode_e4m3(const gda_bf16* q, const gda_bf16* gate, const uint8_t* k_pool,
                    const uint8_t* v_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                    gda_bf16* out, int B, int Hq, int Hkv, int D, float scale, float k_descale,
                    float v_descale, int num_splits, gda_stream_t stream);

/* Prefill / extend gated SDPA (cuDNN FE-OSS "Gated Attention Block (SM107)", Overview
 * stages (4) SDPA with GQA H_q / H_kv and (5) the gate; Fusion knobs: fuse_gate puts
 * O *= sigmoid(GATE) in the SDPA epilogue, after the dead-row select; Forward:
 * return_lse, seq_lens).
 *   q, gate   [B, Sq, Hq, D] bf16          queries and gate (gate NULL: out = RNE_bf16(O))
 *   k, v      [B, Skv, Hkv, D] bf16        keys and values of each sequence
 *   kv_lens   [B] int32 or NULL            valid keys per sequence (0 <= L_b <= Skv; NULL: Skv)
 *   out       [B, Sq, Hq, D] bf16          RNE_bf16(RNE_bf16(O) * RNE_bf16(sigmoid(gate)))
 *   lse       [B, Hq, Sq] float or NULL    natural-log log-sum-exp (-inf for a dead row)
 *   causal    1: key j is visible to query i when j <= i + (L_b - Sq) (the queries are the
 *             last Sq of the L_b positions); 0: every key j < L_b is visible
 *   error_word  device uint32 the kernel ORs GDA_DEVERR_* bits into, or NULL for the
 *             library's own word (gda_prefill_read_error)
 * scale must be finite and > 0 (GDA_ERR_ARG otherwise).
 * D = 256 only (GDA_ERR_UNSUPPORTED otherwise).  All tensors contiguous, device
 * pointers 16-byte aligned (4 for kv_lens / lse / error_word).  One kernel on `stream`,
 * no allocation, no read back; the tensor-map set-up runs on the host per call.
 * The first call on a device also builds the library's 128 KiB BF16 sigmoid table
 * and waits for it (on a stream of its own), so make it before any stream capture:
 * made while `stream` is capturing, it returns GDA_ERR_CAPTURE and enqueues nothing.
 * A query row with no visible key gives O = 0 (out = 0) and lse = -inf. */
int gda_prefill(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k, const gda_bf16* v,
                const int32_t* kv_lens, gda_bf16* out, float* lse, int B, int Sq, int Skv, int Hq, int Hkv,
                int D, float scale, int causal, uint32_t* error_word, gda_stream_t stream);

/* The library's prefill error word (used when gda_prefill gets error_word == NULL) on
 * the current device: synchronises `stream`, stores the bits in *error_word, clears
 * them when `clear` is nonzero; GDA_OK when zero, GDA_ERR_DEVICE otherwise. */
int gda_prefill_read_error(gda_stream_t stream, int clear, uint32_t* error_word);

/* Size of the fixed device scratch area that gda_decode_noalloc uses (16 MiB). */
#define GDA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* gda_decode for callers that must not allocate device memory at all: code that
 * runs where cudaMalloc is forbidden or unsafe -- a serving loop whose memory was
 * budgeted and reserved up front, a custom or pooled allocator that owns all
 * device memory, or a host thread that must never block on the driver's
 * allocator.  The pages have no counterpart for this entry point.
 * Same arguments, layouts and result as gda_decode.  Instead of a workspace it
 * uses one fixed scratch area of GDA_NOALLOC_SCRATCH_BYTES in device memory that
 * the library declares statically: every GPU that loads the library holds it
 * until the process exits, and this call never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *  - Sizes whose gda_workspace_bytes(B, Hq, Hkv, D, num_splits) exceed
 *    GDA_NOALLOC_SCRATCH_BYTES are rejected with GDA_ERR_WORKSPACE (nothing is
 *    enqueued).  With Hq = 16, Hkv = 2, D = 256 that allows B <= 508 in automatic
 *    mode and B * num_splits <= 1020 with explicit splits.
 *  - The first call on each device looks up the scratch's device address and
 *    clears its header on `stream`; make that first call before any stream capture.
 *  - Every call on a device shares the one scratch area, which keeps the last
 *    call's contents: calls that may overlap on the GPU (different streams without
 *    ordering between them) race and give wrong results. */
int gda_decode_noalloc(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k_pool,
                       const gda_bf16* v_pool, const int32_t* kv_indptr, const int32_t* kv_indices,
                       gda_bf16* out, int B, int Hq, int Hkv, int D, float scale, int num_splits,
                       gda_stream_t stream);

/* Grow the internal workspace of the current device for calls up to these sizes,
 * so later gda_decode calls allocate nothing (FreeToken PR #781, Summary:
 * initialise before capture).  Like a growth inside gda_decode it keeps the buffer it
 * replaces allocated, so graphs captured before it stay valid. */
int gda_reserve(int max_B, int Hq, int Hkv, int D, int max_splits);

/* The cluster size (8, 4, 2 or 1 CTAs per (sequence, KV head)) that a decode with
 * `pairs` = B * Hkv (sequence, KV head) pairs and the length bound max_len takes on the
 * current device through the one-kernel path, or 0 when it takes the split path
 * (gda_args.max_len).  A CUDA occupancy query on first use, not a host-only check. */
int gda_small_path_cluster(int64_t pairs, int max_len);

/* The automatic split rule ("chosen per (B, length) from measured time", FreeToken
 * PR #781, Performance), evaluated for B sequences whose longest has lmax positions
 * and whose total is `total`, `heads` segments per sequence (KV heads, or groups of
 * 8 query heads) and `grid` stage-1 CTAs: the uniform split count S (every sequence
 * cut into S equal pieces), or 0 for the stream schedule (equal chunks of the whole
 * batch).  The device applies the same rule to kv_indptr when the caller passes no
 * bound; gda_args.max_len with total_len applies it on the host.  -1 for invalid
 * arguments; min_chunk <= 0 takes the library default (64).  Pure host arithmetic.
 * The rule, measured on GB300 (this function gives it for a BF16 cache):
 *  - the smallest power of two S with 4 S^2 > lmax (about sqrt(lmax / 2)), at least
 *    min_chunk positions each;
 *  - at most one wave of CTAs; when the wave bounds S, the power of two below it if
 *    >= 80 % of the CTAs stay busy, else the bound; below 80 % busy, the stream;
 *  - the stream once each CTA would take >= 3072 positions, or when the longest
 *    sequence is more than 1.25 x the mean.
 * An e4m3 cache streams a position in half the time: its variant of the rule takes
 * 16 S^2 > lmax and moves to the stream from 6144 positions per CTA. */
int gda_auto_splits(int B, int heads, int grid, int min_chunk, int lmax, int64_t total);

/* Byte layout of one decode step's inputs packed into a single block, as
 * gda_decode_step_host takes them: q [B, Hq, D] bf16 at offsets[0] (= 0), gate
 * [B, Hq, D] bf16 at offsets[1], kv_indptr [B + 1] int32 at offsets[2] and
 * kv_indices [nnz] int32 at offsets[3], each part starting on a 256-byte boundary.
 * Returns the block's size in bytes (a multiple of 256), or 0 when a size is out of
 * range (B < 1, Hq < 1, D < 1, nnz < 0) or offsets is NULL.  The pages have no
 * counterpart: the block only lets one step's inputs cross the bus in one copy. */
size_t gda_step_layout(int B, int Hq, int D, int64_t nnz, size_t offsets[4]);

/* One decode step whose inputs and result live in host memory.  It is gda_decode
 * (FreeToken PR #781, Summary: the decode entry point; cuDNN FE-OSS "Gated Attention
 * Block (SM107)", Overview stages (4)-(5)) with the host<->device traffic around it,
 * all enqueued on `stream`:
 *   1. one copy of in_bytes from host_in (the packed block, gda_step_layout) to dev_in
 *      (skipped with GDA_STEP_MAP_IN: the kernels then read host_in in place);
 *   2. gda_decode on the views of dev_in, with the device-resident caches k_pool and
 *      v_pool (GDA_KV_BF16, or GDA_KV_E4M3 codes with k_descale and v_descale as in
 *      gda_args), into dev_out [B, Hq, D] (into host_out with GDA_STEP_MAP_OUT);
 *   3. one copy of dev_out (B * Hq * D bf16) to host_out (skipped with GDA_STEP_MAP_OUT);
 *   4. with synchronize != 0, a wait for the stream, after which host_out holds the
 *      gated output and host_in may be reused.
 * host_in and host_out should be page-locked host memory (cudaHostAlloc, or a pinned
 * torch tensor) for the copies to be asynchronous; pageable memory works, but the
 * runtime then stages it through its own buffers.  dev_in is device memory,
 * 256-byte aligned, at least gda_step_layout(...) bytes; in_bytes must equal that
 * size.  As for gda_decode, every kv_indices entry must name a row of the pools (index
 * contents are not checked on the host).  The host reads the B + 1 kv_indptr values
 * of host_in: kv_indptr[0] != 0, kv_indptr[B] != nnz or a decreasing pair returns
 * GDA_ERR_SHAPE with nothing enqueued; otherwise the longest length and nnz go in as
 * gda_args.max_len and total_len (the one-kernel path or a host-chosen split count
 * where they apply).  The workspace is the library's, as for gda_decode (gda_reserve first
 * to keep the call allocation-free).  Returns the first failing step's status;
 * nothing after a failed step is enqueued.  Without synchronize the caller must not
 * touch host_in or read host_out before the stream has passed this call. */
int gda_decode_step_host(const void* host_in, void* dev_in, size_t in_bytes, const void* k_pool,
                         const void* v_pool, int kv_dtype, float k_descale, float v_descale, gda_bf16* dev_out,
                         void* host_out, int B, int Hq, int Hkv, int D, int64_t nnz, float scale, int num_splits,
                         int flags, int synchronize, gda_stream_t stream);
/* flags of gda_decode_step_host (bitwise or):
 *   GDA_STEP_MAP_IN   the kernels read the inputs from host_in itself over the
 *                     host-device link (no copy; dev_in may be NULL);
 *   GDA_STEP_MAP_OUT  stage 2 writes the result into host_out itself (no copy; dev_out
 *                     may be NULL).
 * A mapped pointer must be page-locked host memory that the device can address
 * (cudaHostAlloc or cudaHostRegister on a system with unified addressing); the call
 * checks that with cudaPointerGetAttributes and returns GDA_ERR_ARG otherwise. */
#define GDA_STEP_MAP_IN 0x1
#define GDA_STEP_MAP_OUT 0x2

/* The step before attention for one decode token per sequence (cuDNN FE-OSS "Gated
 * Attention Block (SM107)", Overview stages (2)+(3), Weights and tables): from the
 * token's projection row [q (Hq*D) | gate (Hq*D) | k (Hkv*D) | v (Hkv*D)] (W_qkvg
 * column blocks Q | GATE | K | V) it writes
 *   q_out[b,h,:]         = rope(rmsnorm(q[b,h,:], w_q_norm))
 *   k_pool[slots[b],h,:] = rope(rmsnorm(k[b,h,:], w_k_norm))
 *   v_pool[slots[b],h,:] = v[b,h,:]
 *   gate_out[b,h,:]      = gate[b,h,:]              (skipped when gate_out is NULL)
 * rmsnorm(x, w) = x / sqrt(mean(x^2) + eps) * w (no norm when w is NULL); rope rotates
 * the first rope_dim dims in the rotate-half convention with cos/sin [B, rope_dim]:
 * out_i = y_i cos_i - y_{i+r/2} sin_i and out_{i+r/2} = y_{i+r/2} cos_{i+r/2} + y_i sin_{i+r/2}
 * for i < r/2 (r = rope_dim); other dims pass through.  FP32 arithmetic, one RNE
 * rounding to bf16.
 *   qgkv      [B, row_stride] bf16, row_stride >= (2 Hq + 2 Hkv) D, a multiple of 8
 *   w_q_norm, w_k_norm  [D] bf16 or NULL; cos_t, sin_t [B, rope_dim] bf16 (rope_dim = 0: none)
 *   slots     [B] int32: each token's slot in the pools; a slot outside [0, num_slots)
 *             is not written
 *   q_out, gate_out [B, Hq, D] bf16; k_pool, v_pool [num_slots, Hkv, D] bf16 (written)
 * D = 256 and rope_dim a multiple of 16 (else GDA_ERR_UNSUPPORTED). */
int gda_qk_norm_rope_kv_write(const gda_bf16* qgkv, int64_t row_stride, const gda_bf16* w_q_norm,
                              const gda_bf16* w_k_norm, float eps, const gda_bf16* cos_t,
                              const gda_bf16* sin_t, int rope_dim, const int32_t* slots,
                              int64_t num_slots, gda_bf16* q_out, gda_bf16* gate_out,
                              gda_bf16* k_pool, gda_bf16* v_pool, int B, int Hq, int Hkv, int D,
                              gda_stream_t stream);

/* Standalone gate, the second half of the unfused path (FreeToken PR #781,
 * Correctness: the fused output equals Torch sigmoid followed by Torch multiply):
 *   out[i] = RNE_bf16( o[i] * RNE_bf16(sigmoid(gate[i])) ),  0 <= i < n.
 * o, gate, out: [n] bf16 device arrays (16-byte aligned; out may alias o). */
int gda_gate(const gda_bf16* o, const gda_bf16* gate, gda_bf16* out, int64_t n,
             gda_stream_t stream);

/* Read (and with clear != 0, reset) the device error word of a workspace -- or of
 * the internal workspace when workspace == NULL.  Synchronises `stream`.  Returns
 * GDA_OK when the word is zero, GDA_ERR_DEVICE otherwise; *error_word gets the bits. */
int gda_read_error(const void* workspace, gda_stream_t stream, int clear, uint32_t* error_word);

/* Stage timing for benchmarks.  After gda_timing_begin(max_calls), each of the next
 * max_calls decode calls (any entry point, any stream) records a CUDA event pair
 * around its stage-1 kernel on its launch stream; stage 2 of those calls then starts
 * after the event instead of overlapping stage 1's tail.  gda_timing_end waits for
 * the recorded events and returns how many stage-1 launches were timed and their
 * summed duration in milliseconds, then releases the events.  Not thread-safe
 * against concurrent decode calls from other threads. */
int gda_timing_begin(int max_calls);
int gda_timing_end(int* n_timed, double* total_ms);

/* Failure-path testing.  The kernels that wait on mbarriers (gda_prefill, and the
 * GDA_VARIANT_TMA stage 1 of the decode) give up a wait after a limit of SM cycles
 * (about two seconds by default), set GDA_DEVERR_TIMEOUT in their error word (the
 * workspace's, or gda_prefill's), wait with the default limit for the copies and MMAs
 * they already started, and return, so the context stays usable and the host reads a
 * typed error instead of a hang (cuDNN FE-OSS "Gated Attention Block (SM107)",
 * Forward: errors are reported, not hung on).  This sets the limit for calls enqueued
 * after it, in this process, on every device: 0 < cycles < the default makes every
 * such pipeline wait poll and give up after `cycles` (a test then sees the timeout
 * path run, and the outputs of those calls are undefined); cycles <= 0 restores the
 * default.  Not for production use.  Returns GDA_OK. */
int gda_debug_wait_limit(int64_t cycles);

/* Static description of a status code. */
const char* gda_status_str(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int gda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDA_H */
