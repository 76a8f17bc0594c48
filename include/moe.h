/*
 * moe.h -- C ABI of libmoe_gb300.so: the single-GPU hot path of an expert-parallel
 * Mixture-of-Experts layer on GB300 (sm_103a).
 *
 * The layer runs four steps (Ultralytics glossary "Expert Parallelism", section "How tokens move
 * across GPUs"; inference guide 6.4 "Data parallelism and expert parallelism", section 3.1):
 *   1. route    -- the router scores every token against every expert and keeps the top k;
 *   2. dispatch -- each token's hidden state is copied once per chosen expert into expert-major
 *                  buffers (here a local permute; there is no all-to-all on one GPU);
 *   3. experts  -- every expert runs its SwiGLU FFN (gate, up, down; guide 6.4 section 2.1) on the
 *                  rows it received, as one grouped GEMM;
 *   4. combine  -- outputs return to their token and are summed with the route weights, plus the
 *                  shared expert (guide 6.4 section 7: the shared expert acts like a routed expert
 *                  every token picks).
 *
 * Conventions common to every entry point
 *   - Pointers named x, w_*, s_*, logits, topk_*, counts, offsets, inv_pos, row_*, xd*, yd, y and
 *     ws are DEVICE pointers owned by the caller; the library never allocates or frees device
 *     memory, never synchronises the stream and never reads results back to the host. Every
 *     device pointer must be 16-byte aligned.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream). The
 *     calls are asynchronous: a return of MOE_OK means the work was enqueued.
 *   - bf16 tensors hold IEEE bfloat16 bit patterns; FP8 tensors hold OCP e4m3 codes (uint8).
 *   - Row-major layouts throughout; "[A, B]" means B is the contiguous dimension.
 *   - Results are deterministic: identical inputs give identical bits (no floating-point atomics).
 *   - A workspace holds one call's intermediates and counters: calls that share a workspace must not
 *     overlap on the GPU (enqueue them on one stream, or order them with events). Calls with their own
 *     workspaces may run concurrently, from any host threads and streams.
 *   - Return value: MOE_OK (0) or a negative status; moe_last_error() then describes it. Argument
 *     errors are detected before any work is enqueued.
 *
 * Shapes supported: 1 <= k <= min(E, 32); E <= 1024; E % n_group == 0; h % 256 == 0;
 * I % 128 == 0; I_shared is 0 or I; T >= 0 (T = 0 is a no-op).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same handle type as cudaStream_t */

/* status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID (-1)     /* null / misaligned pointer, inconsistent sizes or routing shape */
#define MOE_ERR_UNSUPPORTED (-2) /* a shape outside the supported set above */
#define MOE_ERR_WORKSPACE (-3)   /* workspace smaller than moe_workspace_size() */
#define MOE_ERR_CUDA (-4)        /* a CUDA launch or driver call failed (message has the CUDA error) */
#define MOE_ERR_DEVICE (-5)      /* a kernel reported bad data or a timed-out wait (moe_device_status) */

/* scoring functions (moe_config.score) */
#define MOE_SCORE_SOFTMAX 0 /* Mixtral: softmax over all experts, top-k of the logits */
#define MOE_SCORE_SIGMOID 1 /* DeepSeek-V3: sigmoid + selection bias, group-limited top-k */

/* expert arithmetic (moe_config.dtype) */
#define MOE_DTYPE_BF16 0          /* bf16 operands, fp32 accumulation */
#define MOE_DTYPE_FP8_BLOCK128 1  /* e4m3 operands; weights 128x128 fp32 scales, activations 1x128 */
#define MOE_DTYPE_NVFP4 2         /* NVFP4 expert weights (e2m1, e4m3 scale per 16, fp32 per matrix), bf16
                                     activations, fp32 accumulation (TensorRT-LLM "DeepSeek R1 throughput on
                                     Blackwell", "Precision strategy": FP4 MoE weights). h and I must be
                                     multiples of 256 */

/* moe_route flags */
#define MOE_LOGITS_GIVEN 1 /* `logits` is an input: skip the router GEMM */

/* device status bits (moe_device_status) */
#define MOE_STATUS_BAD_EXPERT_INDEX 1 /* a topk_idx entry outside [0, E) was skipped */
#define MOE_STATUS_WAIT_TIMEOUT 2     /* a pipeline wait gave up; outputs of that call are invalid */

/* Physical expert slots of a placement with redundant replicas (inference guide 6.4, sections 5.2-5.3,
 * EPLB). Device arrays. Slot s serves logical expert slot_expert[s] as its replica slot_replica[s];
 * replica i of expert e sits in slot replica_slot[e * max_replicas + i]. An expert's assignments go
 * round-robin over its replicas in token order: the r-th kept token of expert e goes to replica
 * r % replicas[e], row r / replicas[e] of that slot. moe_eplb_plan fills these tables. */
typedef struct {
  int32_t n_slots;              /* E + redundant replicas; at most 1024 */
  int32_t max_replicas;         /* row length of replica_slot */
  const int32_t* slot_expert;   /* [n_slots] */
  const int32_t* slot_replica;  /* [n_slots] */
  const int32_t* replicas;      /* [E] */
  const int32_t* replica_slot;  /* [E, max_replicas] */
} moe_placement;

typedef struct {
  int32_t T;            /* tokens */
  int32_t h;            /* hidden size */
  int32_t E;            /* routed experts */
  int32_t k;            /* experts per token */
  int32_t I;            /* routed expert intermediate size */
  int32_t I_shared;     /* shared expert intermediate size; 0 = no shared expert */
  int32_t n_group;      /* expert groups (1 = no group stage) */
  int32_t topk_group;   /* groups kept per token (Mixtral: n_group = topk_group = 1) */
  int32_t score;        /* MOE_SCORE_SOFTMAX | MOE_SCORE_SIGMOID */
  int32_t renormalize;  /* 1: divide the selected weights by their sum */
  float routed_scale;   /* multiplies the routed weights (DeepSeek-V3: 2.5) */
  int32_t dtype;        /* MOE_DTYPE_BF16 | MOE_DTYPE_FP8_BLOCK128 | MOE_DTYPE_NVFP4 */
  float capacity_factor;/* 0: dropless. > 0: every expert keeps at most ceil(capacity_factor * T * k / E)
                           assignments, the earliest tokens first; the rest skip that expert (Ultralytics
                           "Load balancing and capacity": a capacity factor such as 1.25x the fair
                           share; skipped tokens pass through the residual connection) */
  const moe_placement* placement; /* NULL: one slot per expert. Otherwise the expert-major buffers,
                           counts and offsets are per physical slot (n_slots of them) in slot order */
} moe_config;

/* Expert matrices are row-major [rows, cols] with cols the reduction (K) dimension. NVFP4 matrices
 * (MOE_DTYPE_NVFP4, as written by moe_quantize_weights_nvfp4) are three arrays: codes [rows, cols/2]
 * bytes (element 2i in the low nibble of byte i, 2i+1 in the high nibble), block scales [rows, cols/16]
 * e4m3 bytes (passed through the s_* pointers), and one fp32 matrix scale (g_*); element value =
 * e2m1 * e4m3 * matrix scale. */
typedef struct {
  const float* w_router;   /* [E, h] fp32 router weight (no router bias) */
  const float* bias;       /* [E] fp32 selection bias (sigmoid scoring only), or NULL */
  const void* w_gu;        /* [E, 2I, h]: rows [0, I) gate, rows [I, 2I) up; bf16, e4m3 or NVFP4 codes */
  const float* s_gu;       /* FP8: [E, 2I/128, h/128] fp32 block scales; NVFP4: [E, 2I, h/16] e4m3 bytes */
  const void* w_d;         /* [E, h, I] down projection; bf16, e4m3 or NVFP4 codes */
  const float* s_d;        /* FP8: [E, h/128, I/128]; NVFP4: [E, h, I/16] e4m3 bytes */
  const void* w_gu_shared; /* [2I, h] shared expert gate/up, or NULL when I_shared == 0 */
  const float* s_gu_shared;/* FP8: [2I/128, h/128]; NVFP4: [2I, h/16] */
  const void* w_d_shared;  /* [h, I] shared expert down */
  const float* s_d_shared; /* FP8: [h/128, I/128]; NVFP4: [h, I/16] */
  const float* g_gu;       /* NVFP4 only: [E] fp32 matrix scales of w_gu */
  const float* g_d;        /* NVFP4 only: [E] fp32 matrix scales of w_d */
  const float* g_gu_shared;/* NVFP4 only: [1] */
  const float* g_d_shared; /* NVFP4 only: [1] */
} moe_weights;

/* Byte offsets of the intermediates inside a moe_forward workspace (all 256-byte aligned).
 * R = T*k routed rows; R_tot = R + (I_shared > 0 ? T : 0) rows of the expert-major buffers, the
 * last T of which belong to the shared expert. */
typedef struct {
  size_t logits;     /* [T, E] fp32 */
  size_t topk_idx;   /* [T, k] int32 */
  size_t topk_w;     /* [T, k] fp32 */
  size_t counts;     /* [E] int32 */
  size_t offsets;    /* [E + 1] int32 */
  size_t inv_pos;    /* [T, k] int32 */
  size_t row_token;  /* [R] int32 */
  size_t row_weight; /* [R] fp32 */
  size_t xd;         /* [R_tot, h] bf16 or e4m3 */
  size_t xd_scales;  /* FP8: [R_tot, h/128] fp32 */
  size_t hbuf;       /* [R_tot, I] bf16 or e4m3 (SwiGLU product) */
  size_t h_scales;   /* FP8: [R_tot, I/128] fp32 */
  size_t yd;         /* [R_tot, h] bf16 expert outputs (routed rows already route-weighted) */
  size_t router_w3;  /* [3, E, h] bf16: the router weight as three bf16 terms (tensor-core router) */
  size_t scratch;    /* per-call scratch (status word, the grouped GEMMs' tile counters, histograms;
                        for a batch too small to fill the SMs with router tiles, the router's fp32
                        partial sums) */
  size_t total;      /* bytes required */
} moe_ws_layout;

/* Bytes of device workspace every entry point below accepts (one layout serves all of them).
 * Errors: MOE_ERR_INVALID (null pointer or bad config), MOE_ERR_UNSUPPORTED. */
int moe_workspace_size(const moe_config* cfg, size_t* bytes);
int moe_workspace_layout(const moe_config* cfg, moe_ws_layout* layout);

/* Step 1, routing (Ultralytics "How tokens move across GPUs", step 1; TensorRT-LLM "DeepSeek R1
 * throughput on Blackwell", "RouterGEMM mixed I/O" (bf16 in, fp32 out) and "Top-K kernel fusion":
 * groups first, then the top experts inside them, with a bias and a scaling factor; Perplexity "MoE
 * Router": Mixtral routing is the case top-k-group = all groups; the bias only selects, Ultralytics
 * "Load balancing and capacity").
 *   x        [T, h] bf16 activations (unused with MOE_LOGITS_GIVEN)
 *   weights  w_router and bias are read
 *   logits   [T, E] fp32: output of the router GEMM (fp32-accurate: on the tensor cores with the
 *            weight split into three bf16 terms when E >= 128 and E % 32 == 0, on the CUDA cores in
 *            fp32 otherwise), or the input when flags & MOE_LOGITS_GIVEN; may be NULL without the
 *            flag (then kept in ws)
 *   topk_idx [T, k] int32 out: chosen experts, descending selection key, ties to lower index
 *   topk_w   [T, k] fp32 out: route weights (softmax probability or sigmoid score,
 *            renormalised if asked, times routed_scale)
 *   ws       workspace of moe_workspace_size() bytes (ws_bytes); may be NULL with MOE_LOGITS_GIVEN
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
int moe_route(const moe_config* cfg, const void* x, const moe_weights* weights, float* logits, int flags,
              int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Steps 2-3 of the routing aggregation and the dispatch copy (Perplexity "MoE Router": dense
 * dispatch needs the routing information aggregated per expert; guide 6.4 section 3.1 step 2:
 * each token's hidden state is copied k times). Dropless.
 *   x          [T, h] bf16
 *   topk_idx   [T, k] int32, topk_w [T, k] fp32 (from moe_route)
 *   counts     [E] int32 out: rows per expert (at most the capacity when capacity_factor > 0)
 *   offsets    [E + 1] int32 out: exclusive prefix of counts (offsets[E] = T*k when dropless)
 *   inv_pos    [T, k] int32 out: expert-major row of (token, slot); within an expert rows are in
 *              ascending token order
 *   row_token  [T*k] int32 out: token of each row;  row_weight [T*k] fp32 out: its route weight
 *   xd         [R_tot, h] out: rows in expert-major order, then (with a shared expert) the T
 *              token rows for the shared expert. bf16 copies, or e4m3 codes quantised per 1x128
 *              block (Perplexity "Quantization": activations scaled per 128-element vector at
 *              run time) with xd_scales [R_tot, h/128] fp32 (NULL for bf16)
 *   ws         workspace (scratch histograms and the device status word)
 * A topk_idx entry outside [0, E) is skipped and sets MOE_STATUS_BAD_EXPERT_INDEX. An assignment
 * beyond an expert's capacity is dropped: its inv_pos is -1, it has no row, and combine leaves it out.
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
int moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_w,
                 int32_t* counts, int32_t* offsets, int32_t* inv_pos, int32_t* row_token, float* row_weight,
                 void* xd, float* xd_scales, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Dispatch for callers that cannot allocate device memory. No counterpart on the pages: it is
 * moe_dispatch (same arguments and outputs, same kernels) minus the workspace, for callers that
 * cannot give the library a workspace -- an engine whose memory pool owns all of device memory and
 * allows no other allocation, or a plug-in hook that only sees the layer's inputs and outputs
 * (cudaMalloc may also synchronise the whole device, which such callers cannot afford).
 * Its scratch (per-block histograms, 512 KiB) is a static array in the library's own device memory,
 * held by every GPU that loads the library until the process exits. Limits and behaviour:
 *   - (ceil(T / 512) + 1) * E must not exceed 131072 (e.g. E = 256 allows T up to 261632); larger
 *     sizes return MOE_ERR_UNSUPPORTED before any work is enqueued;
 *   - allocates nothing: no cudaMalloc / cudaFree / allocating library routine;
 *   - the first call on a device looks up the array's device address on that device (set-up), so
 *     make that first call before any stream capture; the address belongs to the context current
 *     on the device, so a call that finds another context there (after cudaDeviceReset, or with
 *     another driver context made current) looks it up again, which is again a set-up call;
 *   - every call shares the one array, so calls that overlap on the GPU (other streams, other host
 *     threads) race and must be serialised by the caller;
 *   - a topk_idx entry outside [0, E) is skipped (inv_pos = -1) as in moe_dispatch, but the status
 *     bit is not reported (there is no workspace to hold it).
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
int moe_dispatch_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_w,
                         int32_t* counts, int32_t* offsets, int32_t* inv_pos, int32_t* row_token, float* row_weight,
                         void* xd, float* xd_scales, moe_stream_t stream);

/* Step 3, the experts (guide 6.4 section 2.1: gate, up, down; Perplexity "Roofline / GroupGEMM":
 * g groups of [m_i, k] x [k, n]; Perplexity "Quantization": SiLU, FP8 block scales). One grouped
 * GEMM per projection over the E routed experts plus the shared expert, tiled on the tensor cores:
 *   H  = silu(xd W_gate^T) * (xd W_up^T)          (stored bf16, or e4m3 1x128 for FP8)
 *   yd = (H W_down^T) * row_weight  (routed rows), (H W_down^T) (shared rows), bf16
 * Work is split from the device-side offsets (no host read-back).
 *   xd, xd_scales, offsets, row_weight  from moe_dispatch
 *   yd  [R_tot, h] bf16 out
 *   ws  workspace (holds H)
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
int moe_expert_ffn(const moe_config* cfg, const moe_weights* weights, const void* xd, const float* xd_scales,
                   const int32_t* offsets, const float* row_weight, void* yd, void* ws, size_t ws_bytes,
                   moe_stream_t stream);

/* Step 4, combine (Ultralytics step 4; guide 6.4 section 3.1 step 4 and section 7):
 *   y[t] = bf16( sum_j yd[inv_pos[t, j]] (+ yd[T*k + t] with a shared expert) ),
 * summed in fp32 in slot order and rounded once.
 *   yd [R_tot, h] bf16, inv_pos [T, k] int32, y [T, h] bf16 out.
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
int moe_combine(const moe_config* cfg, const void* yd, const int32_t* inv_pos, void* y, moe_stream_t stream);

/* The whole layer: route -> dispatch -> experts -> combine, intermediates in ws (their places
 * are given by moe_workspace_layout). x [T, h] bf16 in, y [T, h] bf16 out.
 * bf16 layers with a shared expert run it on a second stream (TensorRT-LLM "DeepSeek R1 throughput
 * on Blackwell", multi-stream: it needs only x): the call records an event on `stream` after routing,
 * enqueues the shared expert (rows read from x, written to rows [T*k, T*k + T) of hbuf and yd) on a
 * library-owned stream of the current device (created with two events on first use, kept for the
 * life of the process), and makes `stream` wait for it before the combine. Work enqueued on `stream`
 * after the call therefore sees the whole layer, and the call can be captured into a CUDA graph on
 * `stream`; the routed rows of xd are the only ones dispatch writes on this path.
 * Errors: as the steps above. */
int moe_forward(const moe_config* cfg, const void* x, const moe_weights* weights, void* y, void* ws,
                size_t ws_bytes, moe_stream_t stream);

/* The whole layer as one CUDA graph (Perplexity "CUDA Graph": one graph per batch size removes the
 * per-kernel launch cost; TensorRT-LLM "Runtime optimizations": CUDA graphs with padding to the
 * nearest captured size). moe_graph_create runs moe_forward once eagerly (lazy set-up), then captures
 * moe_forward(cfg, x, weights, y, ws) on `stream` and instantiates it. The graph keeps every pointer:
 * each moe_graph_launch recomputes y from whatever x holds at that time, with the same config.
 * `stream` must not be the legacy default stream. The caller keeps x, y, ws and the weights alive
 * and unmoved until moe_graph_destroy. Launches on one graph must not overlap (shared workspace).
 * Errors: as moe_forward; MOE_ERR_CUDA if capture or instantiation fails. */
typedef struct moe_graph_s* moe_graph;
int moe_graph_create(const moe_config* cfg, const void* x, const moe_weights* weights, void* y, void* ws,
                     size_t ws_bytes, moe_stream_t stream, moe_graph* graph);
int moe_graph_launch(moe_graph graph, moe_stream_t stream);
int moe_graph_destroy(moe_graph graph);

/* Static 128x128 weight quantisation for the FP8 layer (Perplexity "Quantization": weights are
 * quantised statically per 128x128 tile). For each of `batch` row-major [rows, cols] bf16
 * matrices: scale = amax(tile) / 448 (1 for an all-zero tile), code = e4m3(w / scale) rounded to
 * nearest even with saturation. w [batch, rows, cols] bf16; q [batch, rows, cols] e4m3 out;
 * s [batch, rows/128, cols/128] fp32 out. rows and cols must be multiples of 128.
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
int moe_quantize_weights_fp8(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, float* s,
                             moe_stream_t stream);

/* NVFP4 weight quantisation for MOE_DTYPE_NVFP4 layers (TensorRT-LLM "DeepSeek R1 throughput on
 * Blackwell", "Precision strategy": the MoE weights are FP4; the page does not fix the format, this
 * is the NVFP4 layout). For each of `batch` row-major [rows, cols] bf16 matrices: matrix scale g =
 * amax / (6 * 448) in fp32 (1 for an all-zero matrix); per 16 consecutive elements of a row, block
 * scale s = e4m3(amax_block / (6 g)) and codes e2m1(w / (s g)), nearest even with saturation (all zero
 * when s is zero). w [batch, rows, cols] bf16 in; q [batch, rows, cols/2] codes, s [batch, rows, cols/16]
 * e4m3 bytes and g [batch] fp32 out. cols must be a multiple of 256.
 * Errors: MOE_ERR_INVALID, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
int moe_quantize_weights_nvfp4(const void* w, int64_t batch, int64_t rows, int64_t cols, void* q, void* s,
                               float* g, moe_stream_t stream);

/* EPLB placement plan (inference guide 6.4, sections 5.2-5.3), on the host: n_redundant extra replicas
 * go one by one to the expert with the largest load per replica (first expert on ties); then every
 * replica, carrying load / replicas, is placed heaviest first (expert order on ties) onto the card with
 * the smallest load that still has a free slot (first card on ties). n_cards cards of
 * (E + n_redundant) / n_cards slots each, card-major slot numbering.
 *   load [E] host in: assignments per expert (e.g. counts of recent steps)
 *   replicas [E], slot_expert [E + n_redundant], slot_replica [E + n_redundant],
 *   replica_slot [E * (n_redundant + 1)] (max_replicas = n_redundant + 1; unused entries -1),
 *   card_load [n_cards] (sum of load / replicas on each card) -- host out.
 * Errors: MOE_ERR_INVALID ((E + n_redundant) % n_cards != 0, NULL). */
int moe_eplb_plan(const int64_t* load, int32_t E, int32_t n_cards, int32_t n_redundant, int32_t* replicas,
                  int32_t* slot_expert, int32_t* slot_replica, int32_t* replica_slot, double* card_load);

/* Load balance of the last step run with a workspace (inference guide 6.4, section 5.1: an
 * expert-parallel step waits for its busiest expert; Ultralytics "Load balancing and capacity": a
 * capacity limit drops the assignments beyond it). Computed on the device from the counts and
 * offsets that the last moe_forward or moe_dispatch with this workspace left in it, and written to
 * `stats`, a caller-owned DEVICE buffer of one moe_balance_stats (16-byte aligned); asynchronous on
 * `stream` like every other call. Under a placement the counts are per physical slot.
 *   max_rows       rows of the busiest expert (slot)
 *   active         experts (slots) with at least one row
 *   kept           rows kept, offsets[S] (T*k when dropless)
 *   dropped        T*k - kept: assignments a capacity limit dropped
 *   max_over_mean  max_rows / (kept / S), rounded once to fp32 (0 when kept == 0); S = E, or n_slots
 * Errors: MOE_ERR_INVALID, MOE_ERR_CUDA. */
typedef struct {
  int32_t max_rows;
  int32_t active;
  int32_t kept;
  int32_t dropped;
  float max_over_mean;
  int32_t reserved[3];
} moe_balance_stats;
int moe_balance(const moe_config* cfg, const void* ws, moe_balance_stats* stats, moe_stream_t stream);

/* Device status word of a workspace: waits for `stream`, then reads the MOE_STATUS_* bits that
 * kernels of earlier calls with this workspace set into *status, and clears them. moe_forward clears
 * the word at its start; the step entry points only add bits, so a new workspace (arbitrary
 * contents) should be cleared once with this call before step calls are checked.
 * Returns MOE_OK if no bit was set, MOE_ERR_DEVICE if some were; errors: MOE_ERR_INVALID,
 * MOE_ERR_CUDA. */
int moe_device_status(const moe_config* cfg, void* ws, int32_t* status, moe_stream_t stream);

/* Failure-detection self-test (no fault, no trap, no endless loop): one thread waits, through the
 * bounded wait that every pipeline wait of the grouped GEMMs uses, on an mbarrier that nothing ever
 * completes. After limit_cycles SM clocks (1 .. 4e9) the wait gives up and records
 * MOE_STATUS_WAIT_TIMEOUT in the status word of ws, which moe_device_status then reports; the kernel
 * returns and the context stays usable. Asynchronous on `stream`.
 * Errors: MOE_ERR_INVALID, MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
int moe_selftest_wait_timeout(const moe_config* cfg, void* ws, size_t ws_bytes, int64_t limit_cycles,
                              moe_stream_t stream);

/* Message of the last non-zero status returned on the calling host thread ("" if none). */
const char* moe_last_error(void);

/* Number of CUDA kernels this library has launched in this process so far (all threads, all
 * devices). Profiling aid: the difference around a region counts the library's launches in it. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
