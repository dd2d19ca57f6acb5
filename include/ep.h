/*
 * libep -- MoE expert-parallel dispatch / combine on one GB300 (sm_103a).
 *
 * C ABI. All pointers named d_* or documented as "device" are CUDA device
 * pointers; everything else is host memory. `stream` is a cudaStream_t passed
 * as void* (NULL = legacy default stream). No function allocates device
 * memory: the caller hands one device workspace to ep_config_create and owns
 * every input and combine output; dispatch outputs are views into that
 * workspace, valid until the next ep_dispatch*, ep_reset or ep_destroy.
 * Dispatch and combine never synchronise the host, so they can be captured
 * into a CUDA graph.
 *
 * The EP ranks are simulated: rank r's receive buffers are partitions of the
 * workspace, and inputs carry all ranks at once as [world_size][...] arrays.
 *
 * Operation definitions come from the MORI-EP User Guide:
 *   section 2 "Configuration" (EpDispatchCombineConfig fields),
 *   section 3 "Operator API" (dispatch(), combine(), reset(),
 *             get_dispatch_src_token_pos()),
 *   section 4 "Standard MoE Compatibility (DeepEP)" (dispatch_standard_moe(),
 *             combine_standard_moe(), convert_dispatch_output(),
 *             convert_combine_input()),
 * and from "Choosing an EP API and backend" (EP paths table: the combine is
 * a gather, in bf16 or f32, and dispatch may quantise; restrictions: OCP
 * E4M3 FP8).
 *
 * Thread safety: a handle is not thread-safe; distinct handles are
 * independent. Errors: every call returns an ep_status; ep_last_error()
 * gives a message for the calling thread's most recent failure.
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EP_MAX_WORLD_SIZE 32   /* simulated ranks per handle */
#define EP_MAX_TOPK 32         /* num_experts_per_token */
#define EP_MAX_EXPERTS 1024    /* world_size * num_experts_per_rank */
#define EP_QUANT_BLOCK 128     /* FP8 block: one f32 scale per 128 elements */

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = -1,    /* bad config, pointer, size or alignment */
    EP_ERR_STATE = -2,          /* call out of order (e.g. combine before dispatch) */
    EP_ERR_CAPACITY = -3,       /* packed standard-MoE rows exceed the configured capacity */
    EP_ERR_INVALID_INDEX = -4,  /* expert id outside [-1, E) (or duplicated, standard MoE) */
    EP_ERR_CUDA = -5,           /* a CUDA runtime call failed; see ep_last_error() */
    EP_ERR_TIMEOUT = -6,        /* a kernel's bounded wait gave up (reported by ep_sync) */
    EP_ERR_WORKSPACE = -7,      /* workspace NULL, misaligned or too small */
    EP_ERR_UNSUPPORTED = -8     /* valid request the library does not implement */
} ep_status;

typedef enum {
    EP_DTYPE_BF16 = 0,
    EP_DTYPE_FP32 = 1,
    EP_DTYPE_FP8_E4M3 = 2,      /* OCP E4M3 (bias 7, max 448, NaN = S.1111.111) */
    EP_DTYPE_FP4_E2M1X2 = 3     /* OCP E2M1 codes, two per byte (even element in the low
                                   nibble); pre-quantised pass-through, H % 32 == 0 */
} ep_dtype;

typedef enum {
    EP_COMBINE_AUTO = 0,        /* bulk for the 2D layout from 8192 source tokens on,
                                   vector otherwise; convert_combine_input: bulk */
    EP_COMBINE_VECTOR = 1,      /* 16-byte vector loads into registers */
    EP_COMBINE_BULK = 2         /* bulk async copies (TMA) into a shared-memory ring; needs
                                   <= 8 rows per token (world_size <= 8, or top-k <= 8
                                   for the packed layout), else the vector kernel runs */
} ep_combine_impl;

typedef enum {
    EP_DISPATCH_AUTO = 0,       /* bulk in copy mode from 8192 source tokens on, vector
                                   otherwise */
    EP_DISPATCH_VECTOR = 1,     /* 16-byte vector loads and stores */
    EP_DISPATCH_BULK = 2        /* copy mode only: bulk async copies (TMA) through a
                                   shared-memory ring, rows <= 48 KB; quantisation always
                                   uses the vector kernel */
} ep_dispatch_impl;

/* The two phases whose launch configuration can be set separately
 * (ep_set_launch_config). */
typedef enum {
    EP_PHASE_DISPATCH = 0,      /* routing layout, dispatch, dispatch_standard_moe,
                                   convert_dispatch_output */
    EP_PHASE_COMBINE = 1        /* combine, combine_standard_moe, convert_combine_input */
} ep_phase;

typedef enum {
    EP_QUANT_NONE = 0,          /* dispatch moves the input bits unchanged */
    EP_QUANT_FP8_E4M3_BLOCK128 = 1, /* bf16 in; E4M3 codes + one f32 scale per 128 elements out */
    EP_QUANT_FP4_E2M1_BLOCK32 = 2   /* bf16 in; packed E2M1 codes (H/2 bytes) + one f32 scale
                                       (amax / 6) per 32 elements out; H % 32 == 0 */
} ep_quant;

/*
 * Mirrors EpDispatchCombineConfig (User Guide, section 2). `rank` is absent:
 * all world_size ranks live in this process. Additions are marked (+).
 */
typedef struct ep_config {
    int32_t world_size;                  /* simulated EP ranks, 1..EP_MAX_WORLD_SIZE */
    int32_t hidden_dim;                  /* H, elements per token */
    int32_t scale_dim;                   /* pass-through scales per token (0 = none); with
                                            FP8 (FP4) quantisation 0 or H/128 (H/32), 4-byte */
    int32_t scale_type_size;             /* bytes per pass-through scale element */
    int32_t max_token_type_size;         /* bytes of the widest combine element (2 or 4) */
    int32_t max_num_inp_token_per_rank;  /* Tmax */
    int32_t num_experts_per_rank;        /* E_r; expert e is owned by rank e / E_r */
    int32_t num_experts_per_token;       /* k (top-k), 1..EP_MAX_TOPK */
    int32_t data_type;                   /* ep_dtype of dispatch input tokens: BF16, FP32 or
                                            FP8_E4M3 (pre-quantised pass-through) */
    int32_t quant_type;                  /* (+) ep_quant; FP8 block quant needs BF16 input and
                                            H % 128 == 0 */
    int32_t combine_dtype;               /* (+) ep_dtype of expert outputs given to combine:
                                            BF16 or FP32 */
    int32_t combine_out_dtype;           /* (+) ep_dtype of combine output: BF16 or FP32 */
    int32_t weighted_combine;            /* (+) 0: plain sum over ranks; 1: weighted sum */
    int32_t standard_moe;                /* (+) layouts the workspace reserves: 0 the 2D
                                            receive layout; 1 the per-expert packed layout
                                            only (dispatch_standard_moe /
                                            combine_standard_moe); 2 both, with the
                                            conversions between them */
    int32_t max_packed_rows_per_rank;    /* (+) the packed pool holds world_size times this
                                            many rows; 0 = the worst case of any routing,
                                            R*Tmax*k + 127*R*E_r rows in all */
    int32_t block_num;                   /* CTAs per launch; <= 0: one wave sized to the GPU */
    int32_t warp_num_per_block;          /* warps per CTA; <= 0: 8 */
    int32_t combine_impl;                /* (+) ep_combine_impl */
    int32_t dispatch_impl;               /* (+) ep_dispatch_impl */
    int32_t use_external_inp_buf;        /* 1: combine reads the caller's expert_out (default);
                                            0: also reserve a registered combine input buffer
                                            (see ep_get_registered_combine_input_buffer) */
} ep_config;

typedef struct ep_handle ep_handle;

/*
 * Dispatch results (User Guide, section 3, dispatch() return values). All
 * pointers are device views into the workspace. cap = world_size * Tmax rows
 * per destination rank; rank r's rows start at r * cap. Only the first
 * recv_num_token[r] rows of rank r are written.
 */
typedef struct ep_dispatch_out {
    void* x;                    /* [R][cap][x_row_bytes] payload: input dtype, E4M3 codes,
                                   or E2M1 codes two per byte */
    void* scales;               /* [R][cap][scale_row_bytes]; NULL when there are none */
    float* weights;             /* [R][cap][k] router weights of the received token */
    int32_t* indices;           /* [R][cap][k] global expert ids of the token (-1 kept) */
    int32_t* recv_num_token;    /* [R] rows received by each rank (device) */
    int32_t* src_token_pos;     /* [R][cap] src_rank * (R * Tmax) + src_token_id */
    int64_t cap;                /* rows per destination rank */
    int64_t x_row_bytes;        /* bytes per payload row */
    int64_t scale_row_bytes;    /* bytes per scale row (0 = none) */
} ep_dispatch_out;

/*
 * Standard-MoE (DeepEP-style) packed layout (User Guide, section 4). Rank r
 * holds one contiguous segment per local expert, in ascending expert order,
 * each padded to a multiple of 128 rows; rows inside a segment are ordered
 * by (source rank, source token). The ranks' regions are consecutive in one
 * pool of pcap rows: rank r's rows are pool rows rank_base[r] ..
 * rank_base[r] + rank_rows[r] - 1, rank_base being the exclusive prefix of
 * rank_rows (device values, written by the dispatch). The pool holds the
 * worst case of every routing by default: world_size * Tmax * k rows (one
 * per (token, slot)) plus 127 padding rows per expert.
 */
typedef struct ep_std_moe_out {
    void* packed_x;                 /* [pcap][H] payload (pool) */
    void* packed_scales;            /* [pcap][H/128] (FP8) or [pcap][H/32] (FP4) f32 with
                                       quantisation, else NULL */
    int32_t* packed_count;          /* [R][E_r] rows per local expert */
    int32_t* packed_src_info;       /* [pcap] src_token_pos encoding; -1 on padding rows */
    int64_t* packed_layout_range;   /* [R][E_r][R] (begin << 32) | count per source rank,
                                       begin relative to the expert segment */
    int32_t* expert_offset;         /* [R][E_r] first row of each expert segment within its
                                       rank's region */
    int32_t* rank_rows;             /* [R] padded rows in use on each rank */
    int32_t* rank_base;             /* [R] first pool row of each rank's region */
    int64_t pcap;                   /* rows in the pool */
    int64_t x_row_bytes;
} ep_std_moe_out;

/* Workspace bytes needed by `cfg` (0 if the config is invalid). Host only. */
size_t ep_workspace_size(const ep_config* cfg);

/*
 * Validate `cfg` and carve `d_workspace` (device, 256-byte aligned, at least
 * ep_workspace_size bytes, owned by the caller for the handle's lifetime).
 * Makes no CUDA call; the first dispatch clears the workspace's counters on
 * its stream. Returns EP_ERR_INVALID_ARG / EP_ERR_WORKSPACE on bad input.
 */
ep_status ep_config_create(const ep_config* cfg, void* d_workspace, size_t workspace_bytes,
                           ep_handle** out_handle);

/* Free the host-side handle (the workspace stays the caller's). NULL is a no-op. */
void ep_destroy(ep_handle* h);

/*
 * dispatch() (User Guide, section 3): route every source token once to each
 * distinct rank owning one of its top-k experts (owner = id / E_r; -1 slots
 * are dropped) and copy its payload, weights, indices and scales there.
 *   x          device [R][Tmax][H], data_type; 16-byte aligned
 *   weights    device [R][Tmax][k] f32
 *   scales     device [R][Tmax][scale_dim * scale_type_size bytes] or NULL
 *              (must be NULL with block quantisation, which computes them)
 *   indices    device [R][Tmax][k] int32 in [-1, R*E_r)
 *   num_tokens host [R], tokens held by each source rank, each <= Tmax
 * Receive rows are ordered by (source rank, source token). Needs the 2D
 * layout (standard_moe 0 or 2). State must be READY; afterwards it is
 * DISPATCHED. An out-of-range expert id is skipped
 * and raises EP_ERR_INVALID_INDEX at the next ep_sync.
 */
ep_status ep_dispatch(ep_handle* h, const void* x, const float* weights, const void* scales,
                      const int32_t* indices, const int32_t* num_tokens, void* stream,
                      ep_dispatch_out* out);

/*
 * combine() (User Guide, section 3; a gather): for each source token,
 * sum the expert-output rows of its copies in ascending destination-rank
 * order in an f32 accumulator starting at +0, weighted by the rank's slot
 * weights when weighted_combine, and round once to combine_out_dtype.
 *   expert_out   device [R][cap][H] combine_dtype, rows in dispatch order; NULL
 *                reads the registered combine input buffer (use_external_inp_buf = 0)
 *   weights      device [R][cap][k] f32 in receive layout (dispatch's weights
 *                output or the caller's), or NULL (then out_weights must be
 *                NULL and weighted_combine 0)
 *   indices      accepted for API parity; the dispatch layout is used
 *   out          device [R][Tmax][H] combine_out_dtype (rows past num_tokens untouched)
 *   out_weights  device [R][Tmax][k] f32 or NULL: the weight row of the copy on
 *                the lowest destination rank (zeros for a token sent nowhere)
 *   call_reset   nonzero: ep_reset after the combine
 * State must be DISPATCHED or COMBINED (2D layout present).
 */
ep_status ep_combine(ep_handle* h, const void* expert_out, const float* weights,
                     const int32_t* indices, void* out, float* out_weights, int32_t call_reset,
                     void* stream);

/*
 * get_registered_combine_input_buffer() (User Guide, section 3; zero-copy
 * mode, use_external_inp_buf = 0): device [R][cap][H] buffer of combine_dtype
 * inside the workspace, valid for the handle's lifetime. Experts write their
 * outputs there (row i of rank r for receive row i) and ep_combine with
 * expert_out == NULL reads it in place. EP_ERR_STATE if the config did not
 * reserve it.
 */
ep_status ep_get_registered_combine_input_buffer(ep_handle* h, void** d_buffer);

/* get_dispatch_src_token_pos() (User Guide, section 3): device [R][cap]. */
ep_status ep_get_dispatch_src_token_pos(ep_handle* h, const int32_t** d_src_token_pos);

/* reset() (User Guide, section 3): back to READY; invalidates dispatch views.
 * Enqueues nothing on `stream`. */
ep_status ep_reset(ep_handle* h, void* stream);

/*
 * dispatch_standard_moe() (User Guide, section 4): routing and copy into
 * the packed per-expert layout in one pass (one row per valid (token, slot),
 * no per-rank deduplication). Same inputs as ep_dispatch. Needs
 * standard_moe = 1 or 2. Capacity overflow raises EP_ERR_CAPACITY at ep_sync and
 * the overflowing rows are not written.
 */
ep_status ep_dispatch_standard_moe(ep_handle* h, const void* x, const float* weights,
                                   const void* scales, const int32_t* indices,
                                   const int32_t* num_tokens, void* stream, ep_std_moe_out* out);

/*
 * combine_standard_moe() (User Guide, section 4): per source token, over its
 * valid slots in (owner rank, slot) order, acc = fmaf(w, y, acc) (weighted)
 * or acc + y, f32 from +0, rounded once to combine_out_dtype.
 *   expert_out  device [pcap][H] combine_dtype, in the packed pool's rows
 *   weights     device [R][Tmax][k] f32 source-side router weights (NULL if unweighted)
 *   indices     accepted for API parity; the packed layout is used
 *   out         device [R][Tmax][H]
 * Needs a packed layout (ep_dispatch_standard_moe or ep_convert_dispatch_output).
 */
ep_status ep_combine_standard_moe(ep_handle* h, const void* expert_out, const float* weights,
                                  const int32_t* indices, void* out, int32_t call_reset,
                                  void* stream);

/*
 * convert_dispatch_output() (User Guide, section 4): build the packed layout
 * from the 2D receive buffers of the preceding ep_dispatch.
 *   dispatch_x        device [R][cap][H] (normally ep_dispatch_out.x)
 *   dispatch_indices  device [R][cap][k] (normally ep_dispatch_out.indices)
 * The result equals ep_dispatch_standard_moe on the same inputs. FP8 scales
 * are carried along when the dispatch quantised. Needs standard_moe = 2.
 */
ep_status ep_convert_dispatch_output(ep_handle* h, const void* dispatch_x,
                                     const int32_t* dispatch_indices, void* stream,
                                     ep_std_moe_out* out);

/*
 * convert_combine_input() (User Guide, section 4): from packed expert
 * outputs, build the 2D combine input: receive row i of rank r gets the
 * unweighted f32 sum, over the token's slots owned by r in ascending slot
 * order, of their packed rows, rounded once to combine_dtype.
 *   packed_y    device [pcap][H] combine_dtype, in the packed pool's rows
 *   combine_in  device [R][cap][H] combine_dtype (rows past recv_num_token untouched)
 * Needs both layouts (ep_dispatch, then ep_convert_dispatch_output). Runs
 * the bulk-copy kernel unless the combine phase is set to EP_COMBINE_VECTOR
 * (or top-k > 8); both give the same bits. A bounded wait that gives up sets
 * the timeout bit reported by ep_sync.
 */
ep_status ep_convert_combine_input(ep_handle* h, const void* packed_y, void* combine_in,
                                   void* stream);

/*
 * Launch configuration of one phase (ep_phase) for the calls that follow:
 * `impl` is an ep_dispatch_impl (EP_PHASE_DISPATCH) or ep_combine_impl
 * (EP_PHASE_COMBINE); block_num and warp_num_per_block as in ep_config
 * (<= 0: automatic; at most 8 warps). The User Guide, section 6 (Launch
 * Configuration) lets each call override block_num / warp_per_block, and
 * section 10 (Tuning) reads per-shape launch parameters from tuning files
 * at run time; a binding does both through this setter. Results do not
 * depend on the launch configuration. Host only; any state. Errors:
 * EP_ERR_INVALID_ARG for an unknown phase or impl or more than 8 warps.
 */
ep_status ep_set_launch_config(ep_handle* h, int32_t phase, int32_t impl, int32_t block_num,
                               int32_t warp_num_per_block);

/* The phase's current launch configuration (as set above, or from ep_config). */
ep_status ep_get_launch_config(const ep_handle* h, int32_t phase, int32_t* impl,
                               int32_t* block_num, int32_t* warp_num_per_block);

/*
 * (+) Self-test of failure detection: launches one kernel that waits on a
 * barrier nothing completes. Its bounded wait gives up after about one
 * second, sets the handle's timeout flag and returns normally (no trap or
 * fault), so the next ep_sync reports EP_ERR_TIMEOUT exactly as for a bulk
 * kernel whose copies never arrived, and the handle stays usable. Async.
 */
ep_status ep_selftest_bounded_wait(ep_handle* h, void* stream);

/*
 * (+) Wait for `stream`, then report and clear device-detected errors
 * (EP_ERR_INVALID_INDEX, EP_ERR_CAPACITY) raised by earlier launches.
 */
ep_status ep_sync(ep_handle* h, void* stream);

/* (+) Message for the calling thread's last failed call ("" if none). */
const char* ep_last_error(void);

/*
 * ---------------------------------------------------------------------------
 * One EP rank per workspace, with split send / receive phases (MORI-EP User
 * Guide, section 3, "Split dispatch/combine (send + recv)": dispatch_send()
 * returns the dispatch outputs, dispatch_recv() completes the receive side;
 * combine_send() returns the combine outputs, combine_recv() completes
 * them; section 1, the intra-node kernel type, where ranks exchange tokens
 * over peer-to-peer links).
 *
 * Each rank (a process, or a handle in one process) owns one workspace of
 * ep_rank_workspace_size bytes, created with the same ep_config on every
 * rank (world_size = number of ranks; standard_moe must be 0). The ranks'
 * workspaces are carved identically, and each handle is given every rank's
 * workspace as a device pointer (ep_rank_set_peers): its own, other handles'
 * in the same process, or peers' memory mapped into this process (CUDA IPC
 * or fabric handles; the library maps nothing itself). Results equal those
 * of the single-workspace calls: rank r's receive rows, src_token_pos and
 * combine outputs are rank r's part of ep_dispatch / ep_combine on the
 * whole group's inputs.
 *
 * Phases. The send calls read and write only the rank's own workspace and
 * inputs; the receive calls read the peers' workspaces. The caller orders
 * them: every rank's dispatch_send (and combine_send) must have completed
 * before any rank's dispatch_recv (combine_recv) starts, and every rank's
 * dispatch_recv before any rank's next dispatch_send; e.g. each rank
 * synchronises its stream, then all ranks meet at a host barrier. No kernel
 * waits on another rank. State per handle: READY -dispatch_send-> SENT
 * -dispatch_recv-> DISPATCHED -combine_send-> COMBINE_SENT -combine_recv->
 * COMBINED -ep_rank_reset (or call_reset)-> READY; other orders return
 * EP_ERR_STATE.
 * ---------------------------------------------------------------------------
 */
typedef struct ep_rank_handle ep_rank_handle;

/* Workspace bytes of one rank for `cfg` (0 if invalid or standard_moe = 1). */
size_t ep_rank_workspace_size(const ep_config* cfg);

/*
 * A handle for rank `rank` in [0, world_size) over `d_workspace` (device,
 * 256-byte aligned, owned by the caller). Makes no CUDA call. With
 * world_size 1 the handle is its own only peer; otherwise call
 * ep_rank_set_peers before the first receive phase.
 */
ep_status ep_rank_create(const ep_config* cfg, int32_t rank, void* d_workspace,
                         size_t workspace_bytes, ep_rank_handle** out_handle);

/* Free the host-side handle. NULL is a no-op. */
void ep_rank_destroy(ep_rank_handle* h);

/*
 * peer_workspaces: host array [world_size] of device pointers, entry r the
 * workspace of rank r as this process sees it; entry `rank` must be this
 * handle's own workspace. State must be READY.
 */
ep_status ep_rank_set_peers(ep_rank_handle* h, void* const* peer_workspaces);

/*
 * dispatch_send(): route this rank's tokens and stage them for the ranks
 * that own their experts.
 *   x, weights, scales, indices  device [Tmax][...] of this rank only, as
 *                                ep_dispatch's inputs for one source rank
 *   num_tokens                   tokens held by this rank, <= Tmax
 *   out                          (optional) views of this rank's receive
 *                                buffers: [cap][...] rows, cap = world_size *
 *                                Tmax, recv_num_token [1]; valid after
 *                                dispatch_recv
 * Each token is read once (and quantised once) into the rank's send buffers.
 */
ep_status ep_dispatch_send(ep_rank_handle* h, const void* x, const float* weights,
                           const void* scales, const int32_t* indices, int32_t num_tokens,
                           void* stream, ep_dispatch_out* out);

/*
 * dispatch_recv(): pull this rank's receive rows from every rank's send
 * buffers, ordered by (source rank, source token), and write recv_num_token
 * and src_token_pos (src_rank * (world_size * Tmax) + src_token_id).
 */
ep_status ep_dispatch_recv(ep_rank_handle* h, void* stream);

/*
 * combine_send(): expose this rank's expert outputs to the ranks whose
 * tokens they belong to.
 *   expert_out   device [cap][H] combine_dtype, rows in receive order; NULL:
 *                the experts wrote ep_rank_get_registered_combine_input_buffer
 *   weights      device [cap][k] f32 in receive layout (dispatch's weights
 *                output or the caller's), or NULL; give weights on every
 *                rank or on none
 *   out          device [Tmax][H] combine_out_dtype, this rank's tokens
 *   out_weights  device [Tmax][k] f32 or NULL (needs weights)
 * out and out_weights are written by combine_recv.
 */
ep_status ep_combine_send(ep_rank_handle* h, const void* expert_out, const float* weights,
                          void* out, float* out_weights, void* stream);

/*
 * combine_recv(): for each of this rank's tokens, read its rows from the
 * ranks holding them and reduce them in ascending rank order, f32 from +0,
 * weighted as ep_combine; call_reset nonzero: back to READY afterwards.
 */
ep_status ep_combine_recv(ep_rank_handle* h, int32_t call_reset, void* stream);

/* reset() for a rank handle: back to READY. Enqueues nothing. */
ep_status ep_rank_reset(ep_rank_handle* h);

/* Device [cap][H] combine_dtype buffer inside the rank's workspace that peers
 * read in combine_recv (zero-copy when the experts write it directly). */
ep_status ep_rank_get_registered_combine_input_buffer(ep_rank_handle* h, void** d_buffer);

/* get_dispatch_src_token_pos() of this rank: device [cap]; after dispatch_recv. */
ep_status ep_rank_get_dispatch_src_token_pos(ep_rank_handle* h, const int32_t** d_src_token_pos);

/* Wait for `stream`, then report and clear device-detected errors (an expert
 * id outside [-1, E) in this rank's indices: EP_ERR_INVALID_INDEX). */
ep_status ep_rank_sync(ep_rank_handle* h, void* stream);

/*
 * Routing layout with no device allocation. The pages have no counterpart:
 * this is the layout half of dispatch on its own, for callers that cannot
 * call cudaMalloc -- plugins and embedded engines whose host application has
 * reserved all device memory in its own pool (one more allocation fails or
 * fragments it), and code paths that must not enter a device allocator. It
 * allocates nothing (no cudaMalloc/cudaFree, no allocating library call):
 * its scratch is one static device array of EP_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until the process exits.
 *   indices         device [R][Tmax][k] int32 in [-1, R*E_r)
 *   num_tokens      host [R], each <= Tmax
 *   recv_num_token  device [R] out
 *   src_token_pos   device [R][R*Tmax] out (first recv_num_token[r] rows written)
 *   slot_map        device [R][Tmax][R] out: receive row of token (s,t) on rank r, or -1
 *                   (tokens past num_tokens untouched)
 *   error_flags     device int32 out or NULL: nonzero if an expert id outside
 *                   [-1, E) was skipped
 * Results equal those of ep_dispatch (same kernel, same order). Limit:
 * world_size * Tmax <= EP_NOALLOC_MAX_TOKENS, else EP_ERR_INVALID_ARG with a
 * message. Each call looks up the array's device address with its device
 * current (the first call on a device does this set-up); a call made while
 * its stream is being captured reuses the address found by an earlier call,
 * so make the first call before any stream capture. Under CUDA's lazy
 * module loading (the default) the array is committed on the device by that
 * first call, so it can need 2.3 MiB of free device memory once: make one
 * warm-up call before the host application reserves its memory pool; later
 * calls take no device memory. Every call shares the array and it keeps the
 * last call's contents; each call clears what must start at zero. Calls
 * that overlap on the GPU race on the array: serialise them.
 */
#define EP_NOALLOC_MAX_TOKENS 65536
#define EP_NOALLOC_SCRATCH_BYTES 2433280
ep_status ep_routing_layout_noalloc(int32_t world_size, int32_t max_num_inp_token_per_rank,
                                    int32_t num_experts_per_rank, int32_t num_experts_per_token,
                                    const int32_t* indices, const int32_t* num_tokens,
                                    int32_t* recv_num_token, int32_t* src_token_pos,
                                    int32_t* slot_map, int32_t* error_flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
