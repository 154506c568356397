/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact softmax attention library.
 *
 * The operation (FlashAttention-4 summary, papercache.org, section 2.1; the
 * FlashAttention explainer, wq-win.github.io, section 2): for every batch entry b
 * and query head h,
 *
 *     S = scale * Q K^T + mask,   P = softmax(S) row by row,   O = P V,
 *     LSE_i = ln sum_j exp(S_ij)            (natural log, of the scaled scores)
 *
 * computed tile by tile with the online-softmax (m, l, u) merge so that S and P
 * never reach device memory; and its gradient (same section 2.1):
 *
 *     D = rowsum(dO o O),  dP = dO V^T,  dS = P o (dP - D),
 *     dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q,
 *
 * with P rebuilt from the saved LSE (recomputation: FlashAttention notes,
 * xwysyy.cn, "Recomputation").
 *
 * Masks: causal means query i sees key j only when j <= i. Grouped-query
 * attention: query head h reads KV head h / (H_q / H_kv); dK and dV of a KV head
 * are summed over the query heads that read it.
 *
 * Data types and layouts. q, k, v, o, dout, dq, dk, dv are bf16 (raw 16-bit
 * storage, passed as void*), row-major and contiguous, head dimension innermost:
 *   fixed length (seqlens == NULL):
 *       q, o, dout, dq : [B, N_q, H_q, d]     k, v, dk, dv : [B, N_k, H_kv, d]
 *       lse            : float [B, H_q, N_q]
 *   packed variable length (seqlens != NULL):
 *       seqlens        : device int32 cu_seqlens[B + 1], cu_seqlens[0] = 0,
 *                        non-decreasing; sequence s owns rows
 *                        cu_seqlens[s] .. cu_seqlens[s+1]-1 of q AND of k/v
 *                        (self-attention: one offset array for both)
 *       B              : number of sequences
 *       N_q = N_k      : total packed rows T = cu_seqlens[B]
 *       q, o, dout, dq : [T, H_q, d]          k, v, dk, dv : [T, H_kv, d]
 *       lse            : float [H_q, T]
 *   Supported head dimensions: d = 64 and d = 128. Every pointer must be 16-byte
 *   aligned (tensor-memory-accelerator copies need it).
 *
 * Ownership and execution. The caller allocates and owns every buffer; the
 * library never frees caller memory. Apart from attn_bwd's caller-provided
 * workspace, the library's own device memory is small and kept until the process
 * exits:
 *   - one error word per device;
 *   - the forward's packed-input plan buffer per (device, stream);
 *   - the forward's balanced tile lists per causal shape (see attn_fwd).
 * Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). The only host synchronisations are the first-time
 * set-ups named at each call.
 *
 * CUDA graphs. Every call only enqueues work on `stream`, so it can be captured
 * into a CUDA graph and replayed, with new contents in the same buffers. Make
 * these calls outside capture: the first call of the library on a device, and
 * the first packed forward call on a stream.
 *
 * Errors. Argument errors are detected on the host before anything is launched
 * and return a non-zero attn_status; no exception crosses the ABI. A launch
 * failure returns ATTN_ERR_CUDA. Device-side pipeline waits are bounded: if one
 * ever runs out of time the kernel records ATTN_ERR_TIMEOUT in the device error
 * word and returns; attn_check() reports (and clears) it.
 *
 * Packed offsets are device data the host does not read. The kernels clamp every
 * sequence they decode into the T = N_q packed rows (rows
 * [clamp(cu[s], lo, T), clamp(cu[s+1], start, T)), lo = 0 or the previous
 * sequence's end), so no read or write leaves the caller's buffers whatever the
 * array holds. An array that is not 0, non-decreasing, ..., T is reported as
 * ATTN_ERR_SEQLENS through the device error word (attn_check); the results of
 * such a call are undefined, and rows that no clamped sequence covers are not
 * written.
 *
 * Device resets. The library caches per-device state (the error word's address,
 * the plan buffers and balanced lists above). Calls made after cudaDeviceReset
 * (or any other teardown of the device's primary context) in the same process
 * are unsupported.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* identical to cudaStream_t */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL_PTR = 1,             /* a required pointer is NULL */
  ATTN_ERR_ALIGNMENT = 2,            /* a tensor pointer is not 16-byte aligned */
  ATTN_ERR_UNSUPPORTED_HEADDIM = 3,  /* head dimensions not supported (see each call) */
  ATTN_ERR_BAD_SHAPE = 4,            /* a size is negative, too large, or inconsistent */
  ATTN_ERR_GQA_RATIO = 5,            /* H_q not a positive multiple of H_kv */
  ATTN_ERR_CAUSAL_SHAPE = 6,         /* causal with N_q != N_k (alignment undefined) */
  ATTN_ERR_WORKSPACE = 7,            /* workspace NULL or smaller than required */
  ATTN_ERR_CUDA = 8,                 /* a CUDA runtime call or launch failed */
  ATTN_ERR_TIMEOUT = 9,              /* a device-side bounded wait ran out */
  ATTN_ERR_NO_DEVICE = 10,           /* no usable CUDA device */
  ATTN_ERR_UNSUPPORTED_DEVICE = 11,  /* device is not sm_103 (GB300-class) */
  ATTN_ERR_SEQLENS = 12              /* cu_seqlens is not 0, non-decreasing, ..., N_q */
} attn_status;

/*
 * Forward pass: writes O (bf16) and LSE (fp32, natural log) for every query row.
 * scale is the score multiplier alpha (1/sqrt(d) in the usual definition; any
 * finite value is accepted). A query row that sees no key (only possible with
 * empty sequences) gets O = 0 and LSE = -inf.
 * FlashAttention-4 summary, sections 2.1 (definition), 3.1.2 (pipeline),
 * 3.1.4 (online softmax with conditional rescaling), 3.3 (work tiles are taken
 * longest first).
 *
 * Packed inputs: the call first launches a one-CTA planning kernel that orders
 * the sequences longest first and zeroes a tile counter. It writes into a
 * library-owned device buffer (cudaMalloc'd on the first packed call on each
 * device and stream, kept until the process exits; a later call with more
 * sequences than the buffer holds synchronises that stream once and
 * reallocates it). Make the first packed call on a stream outside stream
 * capture. With more work tiles than SMs the forward then runs one CTA per SM,
 * and each CTA claims its next work tile from that counter when it is ready
 * for one, so the CTAs share unequal sequences evenly; which CTA computes a
 * tile does not change its results.
 *
 * Fixed-length causal shapes with long work tiles run on a persistent grid whose
 * CTAs take their tiles from a balanced list built on the host. The first call
 * with a new (shape, device) builds it, copies it into a library-owned device
 * buffer (cudaMalloc; the call synchronises its stream once) and keeps it until
 * the process exits; later calls reuse it. A first call made while the stream is
 * being captured, or after 256 shapes already hold a list, builds nothing and
 * runs one CTA per work tile instead (same results, slower).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
             const int* seqlens, float scale, attn_stream_t stream);

/*
 * Forward pass with separate head dimensions for queries/keys (d_qk) and for
 * values/outputs (d_v): S = scale * Q K^T contracts over d_qk, O = P V has d_v
 * columns. The FlashAttention-4 summary (experimental setup) benchmarks the
 * (192, 128) head dimensions of the DeepSeek V3 architecture besides equal ones.
 * Supported pairs: (64, 64), (128, 128), (192, 128); anything else returns
 * ATTN_ERR_UNSUPPORTED_HEADDIM. Layouts as for attn_fwd with d replaced by d_qk
 * in q and k and by d_v in v and o: q [B, N_q, H_q, d_qk], k [B, N_k, H_kv, d_qk],
 * v [B, N_k, H_kv, d_v], o [B, N_q, H_q, d_v] (packed: [T, H, d_*]). Everything
 * else (lse, masks, packed inputs, errors, ownership, streams) is as for
 * attn_fwd, which is this call with d_qk = d_v = d. attn_bwd_dims is the
 * matching backward pass.
 */
int attn_fwd_dims(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v, int causal,
                  const int* seqlens, float scale, attn_stream_t stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (0 on invalid
 * sizes). Arguments mean what they mean for attn_bwd; `varlen` is non-zero when
 * attn_bwd will be given a cu_seqlens array (then N_q is the packed row count).
 * The workspace holds the fp32 dQ accumulator [rows, H_q, d], D = rowsum(dO o O)
 * (laid out like lse), in deterministic mode one ordering semaphore per
 * (query tile, query head) plus a work counter, and for packed inputs the
 * order in which the backward walks the sequences (2 B + 1 ints).
 */
size_t attn_bwd_workspace_bytes(int B, int H_q, int H_kv, int N_q, int N_k, int d, int varlen,
                                int deterministic);

/*
 * Backward pass: given q, k, v, the forward outputs o and lse, and the output
 * gradient dout, writes dq [like q], dk and dv [like k] (bf16, overwritten, not
 * accumulated into). `workspace` is caller-owned device memory of at least
 * attn_bwd_workspace_bytes(...) bytes, 256-byte aligned; its contents on entry
 * do not matter and are undefined on return. With deterministic != 0 the dQ
 * reduction across key tiles runs in a fixed order, so dq, dk and dv are
 * bit-identical across runs with the same inputs on the same device. That order
 * (shortest processing time first) is chosen from the shape:
 *   - causal: walk up from the diagonal;
 *   - equal query and key lengths and at most 32 key tiles per (batch, KV head)
 *     (and at most one per SM): a rotated walk;
 *   - otherwise: ascending key tiles.
 * The rotated walk needs all key tiles of a (batch, KV head) resident together.
 * Kernels on other streams that hold SMs for longer than the wait limit
 * (attn_set_wait_limit) make such a call end with ATTN_ERR_TIMEOUT recorded.
 * FlashAttention-4 summary, sections 2.1 (gradients), 3.2.2 (pipeline),
 * 3.2.4 (deterministic mode).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv,
             int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
             const int* seqlens, float scale, int deterministic,
             void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Backward pass with separate head dimensions for queries/keys (d_qk) and for
 * values/outputs (d_v), the gradient of attn_fwd_dims: layouts as there, with
 * dq like q [.., H_q, d_qk], dk like k [.., H_kv, d_qk], dv like v
 * [.., H_kv, d_v], o and dout [.., H_q, d_v]. Supported pairs: (64, 64),
 * (128, 128), (192, 128); anything else returns ATTN_ERR_UNSUPPORTED_HEADDIM.
 * attn_bwd is this call with d_qk = d_v = d. The FlashAttention-4 summary
 * (experimental setup) benchmarks the (192, 128) head dimensions of the
 * DeepSeek V3 architecture.
 *
 * At d_qk = 192 the main kernel runs in two passes over the key tiles: the
 * first accumulates dV and the query/key head columns 0-127 of dK and dQ, the
 * second columns 128-191; both recompute S and dP (the tensor memory of one
 * SM holds dV, dK, S and dP/dQ for 128 columns, not 192). Everything else
 * (workspace, determinism, errors, streams) is as for attn_bwd, with the
 * workspace size from attn_bwd_dims_workspace_bytes.
 */
size_t attn_bwd_dims_workspace_bytes(int B, int H_q, int H_kv, int N_q, int N_k, int d_qk,
                                     int d_v, int varlen, int deterministic);
int attn_bwd_dims(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv,
                  int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v, int causal,
                  const int* seqlens, float scale, int deterministic,
                  void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Size of the library's own scratch buffer used by attn_bwd_noalloc: 64 MiB on
 * every GPU that loads the library, held until the process exits.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate device
 * memory when they run the backward pass (a plugin whose host program owns all
 * device memory through its own pool and offers no allocator; a latency-critical
 * loop where cudaMalloc / cudaFree would stall on an implicit device
 * synchronisation). The pages this library follows have no counterpart of this
 * call: it is an interface convenience, not part of the method.
 *
 * Arguments, layouts, results and determinism are those of attn_bwd; inputs and
 * outputs are still caller-owned. The scratch is a fixed
 * ATTN_NOALLOC_SCRATCH_BYTES buffer inside the library's device code; nothing is
 * allocated. Problems whose attn_bwd_workspace_bytes(...) exceeds that size are
 * rejected with ATTN_ERR_WORKSPACE before anything is launched. Every call looks
 * up the buffer's device address on the current device (a lookup, no
 * allocation); the first lookup on a device loads the library's device code
 * there, so make the first call on a device before any stream capture. All calls on
 * a device share the one buffer and it keeps the last call's contents (the call
 * clears what must start at zero), so calls whose kernels overlap on the GPU
 * (different streams, or different host threads) race on it and give wrong
 * results: serialise them.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv,
                     int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                     const int* seqlens, float scale, int deterministic, attn_stream_t stream);

/*
 * Synchronises `stream`, then returns the first failure a kernel of this library
 * on the current device recorded since the last check (and clears the record):
 * ATTN_ERR_TIMEOUT for a timed-out wait, ATTN_ERR_SEQLENS for an inconsistent
 * packed-sequence offset array; ATTN_ERR_CUDA if the stream reports an error;
 * else ATTN_OK.
 */
int attn_check(attn_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(int status);

/*
 * Test hook for the FMA-pipe exp2 used inside the forward kernel: y[i] =
 * 2^x[i] computed with mode 0 = the hardware ex2.approx instruction, mode 1 =
 * the degree-3 polynomial emulation (FlashAttention-4 summary, section 3.1.3).
 * x and y are device float arrays of n elements.
 */
int attn_debug_exp2(const float* x, float* y, int n, int mode, attn_stream_t stream);

/*
 * Measurement hook for the forward's conditional rescaling (FlashAttention-4
 * summary, section 3.1.4; the Korean FA-4 review reports about 10x fewer
 * rescales than rescaling whenever the max grows). In a library built with
 * ATTN_COUNT_RESCALE=1 the forward kernels count, over all calls since the last
 * reset, out[0] the (warp, key tile) softmax steps after each row's first key
 * tile, out[1] those steps in which the warp rescaled O and l, out[2] the rows
 * whose exponent bias moved, out[3] the row steps counted. Writes the four
 * counts into out (4 entries) and returns 4, clearing them when reset != 0;
 * returns 0 without touching out in the shipped build, which has no counters;
 * a negative attn_status on failure. Synchronous (waits for the device).
 */
int attn_debug_rescale_stats(unsigned long long* out, int reset);

/*
 * Failure-path test hooks. They exercise the bounded device-side waits without
 * faulting, trapping or hanging the GPU.
 *
 * attn_debug_inject(fault) sets a process-wide injected fault for later
 * launches: ATTN_FAULT_NONE restores normal operation; ATTN_FAULT_SKIP_DQ_RELEASE
 * makes the first work item of a deterministic attn_bwd never release its dQ
 * ordering semaphores, so the key tiles after it give up waiting once the wait
 * limit is spent and the call ends with ATTN_ERR_TIMEOUT recorded (its gradients
 * are then not valid). Returns ATTN_ERR_BAD_SHAPE for an unknown fault.
 *
 * attn_debug_stall(stream) launches one CTA that waits on an mbarrier nothing
 * arrives at; the wait gives up after the wait limit and records
 * ATTN_ERR_TIMEOUT, which attn_check() then reports.
 */
#define ATTN_FAULT_NONE 0
#define ATTN_FAULT_SKIP_DQ_RELEASE 1
int attn_debug_inject(int fault);
int attn_debug_stall(attn_stream_t stream);

/*
 * Host-only view of the forward's launch plan (FlashAttention-4 summary,
 * section 3.3: work tiles taken longest first), for checking it without a GPU.
 * For the shape of an attn_fwd_dims call (varlen != 0: packed inputs, B
 * sequences of N_q = N_k total rows) on a GPU with n_sm SMs, writes six entries
 *   info[0] mode: 0 one CTA per work tile, 1 persistent grid with CTA c taking
 *           tiles c, c + grid, ..., 2 persistent grid over balanced lists,
 *           3 persistent grid whose CTA c takes tile c first and then claims
 *           the next unclaimed tile of the work list from a counter each time
 *           it is ready for one (packed inputs with more tiles than SMs)
 *   info[1] grid size
 *   info[2] work tiles (two 128-row query tiles each; an upper bound when
 *           packed)
 *   info[3] query heads per L2 section
 *   info[4] m-blocks per batch entry (0 when packed): 256 query rows of one head,
 *           or 128 rows with info[5]
 *   info[5] 1 when a work tile holds the same 128 query rows of two adjacent
 *           query heads of one KV head (causal masks with an even GQA group), so
 *           both its query tiles visit the same key tiles; 0 for 256 rows of one
 *           head
 * and, for mode 2 when lists != NULL and lists_cap >= info[1] + 1 + info[2],
 * the lists: lists[0 .. grid] are the CTAs' start offsets into
 * lists[grid + 1 ..], which hold the work-tile indices of CTA c from
 * lists[grid + 1 + lists[c]] to lists[grid + 1 + lists[c + 1] - 1], in the order
 * the CTA takes them. Work tile v is numbered batch outermost, then L2 section,
 * then m-block (longest first), then query head (or head pair). A real call uses
 * mode 2 only when it can build the list (outside stream capture, at most 256
 * shapes);
 * otherwise it runs mode 0. Nothing is launched and no device is needed.
 * Returns ATTN_OK, or the argument error attn_fwd_dims would return.
 */
int attn_debug_fwd_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d_qk, int d_v,
                        int causal, int varlen, int n_sm, long long* info, int* lists,
                        long long lists_cap);

/*
 * Selects the backward main kernel used at d = 128 by later attn_bwd calls in
 * this process: ATTN_BWD_ONE_CTA (default) runs one CTA per 128-key tile;
 * ATTN_BWD_CTA_PAIR runs the 2-CTA backward of the FlashAttention-4 summary,
 * section 3.2.3 (clusters of two CTAs per 256 keys, M = 256 tcgen05 MMAs with
 * operand B split between the CTAs, half of dS exchanged through distributed
 * shared memory, each CTA reducing 64 rows of every dQ tile). Both give results
 * within the same tolerances; on GB300 the pair kernel is the slower one, so it
 * is kept for measurement. d = 64 always uses the one-CTA kernel. Returns the
 * previous selection, or -1 (and changes nothing) for an unknown value.
 */
#define ATTN_BWD_ONE_CTA 0
#define ATTN_BWD_CTA_PAIR 1
int attn_set_bwd_variant(int variant);

/*
 * Selects the forward kernel used by later attn_fwd / attn_fwd_dims calls in
 * this process at d_qk = d_v = 128: ATTN_FWD_ONE_CTA (default) runs two 128-row
 * query tiles per CTA under the work-list schedule described for attn_fwd;
 * ATTN_FWD_CTA_PAIR runs the M = 256 forward on CTA pairs (FlashAttention-4
 * summary, section 2.2, the 2-CTA tensor-core mode): a cluster of two CTAs owns
 * 512 query rows of one (batch, query head), and one thread issues
 * cta_group::2 MMAs with the keys of S = Q K^T and the head-dimension columns
 * of O += P V split between the CTAs. Both give results within the same
 * tolerances; on GB300 the pair kernel is the slower one, so it is kept for
 * measurement. Other head dimensions always use the one-CTA kernel. Returns the
 * previous selection, or -1 (and changes nothing) for an unknown value.
 */
#define ATTN_FWD_ONE_CTA 0
#define ATTN_FWD_CTA_PAIR 1
int attn_set_fwd_variant(int variant);

/*
 * Sets the cycle budget of every bounded device-side wait for later launches
 * on this process (default about one second of SM clock). Returns the old value.
 */
long long attn_set_wait_limit(long long cycles);

/*
 * Kernel tracing. While enabled (process-wide), every kernel this library
 * launches is bracketed by two CUDA events recorded on the launching stream.
 * attn_profile_read() waits for the recorded events, copies up to
 * `max_records` records (oldest first) and discards everything it has read;
 * it returns the number of records written, or a negative attn_status.
 * Kernel ids: 1 forward, 2 backward pre (D, zeroing), 3 backward main (its first
 * pass at d_qk = 192), 4 backward post (dQ conversion), 5 exp2 test hook, 6 stall
 * test hook, 7 forward planning kernel (packed inputs), 8 forward on CTA pairs
 * (ATTN_FWD_CTA_PAIR), 9 second pass of the backward main kernel (d_qk = 192),
 * 10 backward planning kernel (packed inputs).
 */
typedef struct {
  int kernel;  /* kernel id, see above */
  float ms;    /* elapsed time between the two events */
} attn_profile_record;

int attn_profile_enable(int enable);
int attn_profile_read(attn_profile_record* out, int max_records);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
