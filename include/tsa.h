/*
 * tsa.h -- C ABI of libtsa, topology-scheduled sparse attention for GB300 (sm_103a).
 *
 * Method: "Add topology-derived sparse attention kernel" (triton-lang/kernels#22),
 * Summary; and the port note on that PR's GitHub mirror page ("A port of the Triton
 * kernel merged as triton-lang/kernels#22").  The operations:
 *
 *   tsa_build_schedule      -- causal CSR block schedule from K: sink blocks, local-window
 *                              blocks and top-k blocks by 0D-persistence (elder-rule)
 *                              salience over key-block centroids.
 *   tsa_dense_causal_csr    -- the dense causal CSR (every block j <= i).
 *   tsa_segment_csr         -- the CSR of a segment mask (fixed or listed segment starts).
 *   tsa_build_schedule_ex   -- tsa_build_schedule with the elder rule's tie rule chosen
 *                              (block index, or centroid content).
 *   tsa_block_sums / tsa_build_schedule_from_sums -- the same build in two halves, for keys
 *                              whose lanes are spread over several GPUs.
 *   tsa_scheduled_attention -- forward causal attention that visits, for each 64-token query
 *                              block, only the key blocks in its CSR row (online softmax,
 *                              token-level causal mask in the diagonal block);
 *                              tsa_scheduled_attention_fwd also writes the row log-sum-exp.
 *   tsa_scheduled_attention_backward -- dQ, dK, dV of that attention over the same CSR.
 *
 * Conventions shared by every call:
 *   - Every pointer argument except `salience_sq` is required.  Buffers are DEVICE memory
 *     of the current CUDA device, allocated and owned by the caller; the library never
 *     allocates or frees and keeps no pointer after a call returns.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  The return value reports only what the host can check
 *     before launch.  Problems met on the device (an out-of-range or unsorted col_idx, a
 *     wait that timed out) set a device status word read by tsa_last_device_status().
 *     No kernel traps.
 *   - Dense tensors are contiguous row-major.  A lane is one [S, D] matrix; [B, H, S, D]
 *     input is B*H lanes stored back to back ([S, D] input is B = H = 1).  One CSR is
 *     shared by all lanes.
 *   - A CSR schedule is int32: row_ptr[nb + 1] with row_ptr[0] = 0 and non-decreasing,
 *     col_idx[row_ptr[nb]]; row i lists key blocks j, strictly ascending, 0 <= j <= i.
 *     nb = S / block.  The number of stored blocks (nnz) is row_ptr[nb], on the device.
 */
#ifndef TSA_H_
#define TSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream handle: the same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *tsa_stream_t;

typedef enum {
    TSA_OK = 0,
    TSA_ERR_INVALID_ARGUMENT = 1,  /* null pointer, non-positive size, misaligned, ...      */
    TSA_ERR_UNSUPPORTED = 2,       /* valid request this build does not implement          */
    TSA_ERR_NOT_DEVICE_POINTER = 3,/* a buffer is not device memory                        */
    TSA_ERR_DEVICE_MISMATCH = 4,   /* a buffer lives on another device than the current one */
    TSA_ERR_CAPACITY = 5,          /* col_cap or workspace_bytes too small                 */
    TSA_ERR_CUDA = 6,              /* a CUDA runtime / driver call failed                  */
    TSA_ERR_TIMEOUT = 7,           /* device: a bounded wait gave up (kernel returned)     */
    TSA_ERR_BAD_SCHEDULE = 8,      /* device: a CSR row broke the contract above           */
    TSA_ERR_DEVICE = 9             /* device: another device-side check failed             */
} tsa_status;

typedef enum { TSA_F16 = 0, TSA_BF16 = 1 } tsa_dtype;

/* Human-readable name of a status code (static storage; never NULL). */
const char *tsa_status_string(tsa_status status);

/*
 * Upper bound on the nnz of a topology schedule:
 *   sum_{i=0}^{nb-1} min(i + 1, sink + local_radius + 1 + topk),  nb = ceil(S / block).
 * Size col_idx with at least this many entries for tsa_build_schedule.
 * Returns -1 for invalid arguments (S <= 0, block <= 0, negative counts).
 *
 * Partial last block (here and in tsa_build_schedule, tsa_dense_causal_csr and the attention
 * forward): S need not be a multiple of the block.  There are nb = ceil(S / block) blocks; the
 * last holds the S - (nb-1)*block tokens that exist, its centroid averages those tokens, and
 * attention sees keys k < S only.  The pages do not say; this is the plainest reading.
 */
int64_t tsa_schedule_max_nnz(int64_t S, int64_t block, int64_t sink, int64_t local_radius,
                             int64_t topk);

/*
 * Bytes of device workspace tsa_build_schedule needs for `lanes` lanes of [S, D] keys
 * (per-lane block sums, centroids, the pairwise distance intervals and MST state).
 * Returns 0 for invalid arguments.
 */
size_t tsa_build_schedule_workspace_bytes(int64_t lanes, int64_t S, int64_t D, int64_t block);

/*
 * Topology schedule ("Add topology-derived sparse attention kernel", Summary: sink blocks,
 * local-window blocks and a 0D-persistence-style salience over key-block centroids; the
 * mirror page's port note: the salience is the elder rule and exactly one block scores 0).
 *
 *   K            [lanes, S, D] keys (f16 or bf16 per dtype).
 *   centroids    C[b][d] = (sum_lanes (sum_{t in block b} K)) / (block * lanes), binary64,
 *                both sums sequential in ascending order.
 *   distance     d2(u,v) = sum_d (C[u][d] - C[v][d])^2 in binary64: 32 partial sums over
 *                d = j mod 32 (ascending d, one fused multiply-add per term), then halving
 *                (P_j += P_{j+w}, w = 16, 8, 4, 2, 1).
 *   salience     Kruskal order on edges (d2, min(u,v), max(u,v)); the smaller component is
 *                absorbed, on a size tie the one whose root has the larger index; the
 *                absorbed root gets the edge's d2 (squared merge distance); one block keeps 0.
 *   row i        {j < sink} U {max(0, i - local_radius) .. i} U {topk blocks j <= i of
 *                largest salience, lower j on ties}, all clipped to j <= i, ascending.
 *
 *   row_ptr      out, nb + 1 int32.       col_idx  out, col_cap int32 (>= tsa_schedule_max_nnz).
 *   salience_sq  out, nb binary64 (optional, may be NULL): per-block squared merge distance.
 *   workspace    scratch of >= tsa_build_schedule_workspace_bytes(lanes, S, D, block) bytes,
 *                256-byte aligned; its contents on entry do not matter.
 *
 * Limits: 1 <= block, 1 <= nb = ceil(S/block) <= 4096, 1 <= D <= 1024, lanes >= 1.
 * Errors: INVALID_ARGUMENT, NOT_DEVICE_POINTER, DEVICE_MISMATCH, CAPACITY, UNSUPPORTED
 * (nb or D beyond the limits), CUDA.  The result is bit-identical to the CPU oracle.
 */
tsa_status tsa_build_schedule(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S,
                              int64_t D, int64_t block, int64_t sink, int64_t local_radius,
                              int64_t topk, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                              double *salience_sq, void *workspace, size_t workspace_bytes,
                              tsa_stream_t stream);

/*
 * Tie rule of the elder rule.  TSA_TIE_INDEX is the rule above (ties on edge distance and on
 * component size broken by block index).  TSA_TIE_CONTENT is the fix the mirror page's port
 * note asks for (per-block salience is not permutation-equivariant because a size tie is broken
 * by index; a fix needs a tie-break on centroid content): every tie the index rule breaks by
 * index is broken by the centroid instead -- blocks compare lexicographically over d, each
 * coordinate in IEEE 754 totalOrder (-0 before +0), and only bit-identical centroids fall back
 * to the index.  Edges order by (d2, earlier endpoint, later endpoint) in that block order; on a
 * size tie the root that comes later is absorbed.  Moving whole key blocks then moves each
 * block's salience with it, bit for bit.  The top-k order (salience descending, lower j on
 * ties) is the same under both rules.
 */
typedef enum { TSA_TIE_INDEX = 0, TSA_TIE_CONTENT = 1 } tsa_tie_break;

/*
 * tsa_build_schedule with an explicit tie rule (tsa_build_schedule is this call with
 * TSA_TIE_INDEX).  Same arguments, workspace, limits and errors, plus INVALID_ARGUMENT for an
 * unknown tie_break.  The result is bit-identical to the CPU oracle under the same rule.
 */
tsa_status tsa_build_schedule_ex(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S,
                                 int64_t D, int64_t block, int64_t sink, int64_t local_radius,
                                 int64_t topk, tsa_tie_break tie_break, int32_t *row_ptr,
                                 int32_t *col_idx, int64_t col_cap, double *salience_sq,
                                 void *workspace, size_t workspace_bytes, tsa_stream_t stream);

/*
 * The schedule build in two halves, for keys whose lanes are spread over several GPUs
 * (the schedule is one CSR shared by all lanes, built from the lane-mean centroids).
 *
 * tsa_block_sums: per-lane block sums of this GPU's lanes, the first stage of
 * tsa_build_schedule -- part[l][b][d] = sum over the block's tokens t (ascending) of
 * K[l][b*block + t][d], in binary64, the same value tsa_build_schedule forms internally.
 *   K     [lanes, S, D] f16/bf16, device (this GPU's lanes, contiguous).
 *   part  device buffer of lanes * (S / block) * D doubles, written.
 * Limits and errors as tsa_build_schedule.
 *
 * tsa_build_schedule_from_sums: the rest of tsa_build_schedule_ex from the block sums of ALL
 * lanes: centroid C[b][d] = (sum over l ascending of part[l][b][d]) / (block * lanes), then
 * distances, MST, elder rule, top-k and CSR exactly as there.  Gather every GPU's block sums
 * in global lane order (an all-gather of lanes * nb * D doubles) and call this on each GPU:
 * every GPU gets the CSR, bit for bit, that tsa_build_schedule_ex returns for all the keys
 * on one GPU.  (Summing per-GPU totals instead would re-associate the lane sum.)
 *   part        [lanes][nb][D] binary64, device, read only.
 *   S           nb * block (the sequence length the CSR is for).
 *   workspace   >= tsa_build_schedule_workspace_bytes(lanes, S, D, block) bytes.
 * Other arguments, limits and errors as tsa_build_schedule_ex.
 */
tsa_status tsa_block_sums(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S, int64_t D,
                          int64_t block, double *part, tsa_stream_t stream);
tsa_status tsa_build_schedule_from_sums(const double *part, int64_t lanes, int64_t S, int64_t D,
                                        int64_t block, int64_t sink, int64_t local_radius,
                                        int64_t topk, tsa_tie_break tie_break, int32_t *row_ptr,
                                        int32_t *col_idx, int64_t col_cap, double *salience_sq,
                                        void *workspace, size_t workspace_bytes,
                                        tsa_stream_t stream);

/*
 * Segment schedules ("Add topology-derived sparse attention kernel" mirror page, the later
 * commit on a forget gate's exact zeros feeding the merged CSR kernel: a segment boundary is a
 * CSR schedule the kernel runs with zero error; at S 4096, block 64 fixed 512-token segments
 * visit 288 blocks and 256-token segments 160).
 *
 * Segments begin at token 0 and at each start.  Query token q may attend to key k iff
 * s(q) <= k <= q, s(q) the last segment start <= q.  Row i holds every key block with a key
 * allowed to some query of block i: the run s(block * i) / block .. i.  When every start is a
 * multiple of `block`, attention over this CSR is exactly causal attention within each segment;
 * otherwise the CSR is the smallest block schedule covering the segment mask, and the
 * attention kernel lets tokens see across a boundary that falls inside a block.
 *
 * tsa_fixed_segment_nnz: nnz of fixed segments of segment_tokens tokens (starts at multiples of
 *   segment_tokens); -1 for invalid arguments (S % block != 0, non-positive sizes, nb > 65534).
 * tsa_fixed_segment_csr: that CSR.  col_cap >= tsa_fixed_segment_nnz(...), else CAPACITY.
 * tsa_segment_csr: `starts` is a DEVICE array of n_starts int32 tokens, strictly ascending in
 *   [0, S) (n_starts may be 0: one segment, the dense causal CSR).  Only the longest valid
 *   prefix of `starts` is used; an entry out of order or range sets BAD_SCHEDULE in the device
 *   status word.  nnz is at most nb(nb+1)/2; if it exceeds col_cap the rows are cut to fit and
 *   the status word reports TSA_ERR_DEVICE.
 *
 *   row_ptr out, nb + 1 int32;  col_idx out, col_cap int32.
 * Limits: S % block == 0, nb <= 65534, S < 2^31.  Errors: INVALID_ARGUMENT, CAPACITY,
 * NOT_DEVICE_POINTER, DEVICE_MISMATCH, CUDA.
 */
int64_t tsa_fixed_segment_nnz(int64_t S, int64_t block, int64_t segment_tokens);
tsa_status tsa_fixed_segment_csr(int64_t S, int64_t block, int64_t segment_tokens,
                                 int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                                 tsa_stream_t stream);
tsa_status tsa_segment_csr(int64_t S, int64_t block, const int32_t *starts, int64_t n_starts,
                           int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                           tsa_stream_t stream);

/*
 * Dense causal CSR ("Add topology-derived sparse attention kernel", Summary: "dense causal
 * CSR layout"; Local benchmark: the dense CSR path visits every causal block):
 * row_ptr[i] = i(i+1)/2, row i = 0..i.  nnz = nb(nb+1)/2 (136 at nb 16, 2080 at nb 64).
 *
 *   row_ptr out, nb + 1 int32;  col_idx out, col_cap >= nb(nb+1)/2 int32 (nb = ceil(S/block)).
 * Limits: nb(nb+1)/2 < 2^31.  Errors: INVALID_ARGUMENT, CAPACITY,
 * NOT_DEVICE_POINTER, DEVICE_MISMATCH, CUDA.
 */
tsa_status tsa_dense_causal_csr(int64_t S, int64_t block, int32_t *row_ptr, int32_t *col_idx,
                                int64_t col_cap, tsa_stream_t stream);

/*
 * Scheduled attention forward ("Add topology-derived sparse attention kernel", Summary:
 * forward-only kernel over causal CSR block schedules, [seq, dim] and [batch, heads, seq,
 * dim] inputs sharing one CSR, output in the input dtype; mirror page port note: running
 * maximum and denominator, rescale by exp(m_prev - m_new)).
 *
 * For lane l and query token q of query block i = q / 64:
 *   O[l][q] = sum_{k : k/64 in row i, k <= q} softmax_k(scale * <Q[l][q], K[l][k]>) V[l][k]
 * accumulated in fp32 from f16/bf16 inputs and rounded to the input dtype.  A query with
 * no allowed key gets O = 0.
 *
 *   Q, K, V  in,  [B*H, S, D] of `dtype`, 16-byte aligned.
 *   O        out, same shape and dtype (must not alias Q, K or V).
 *   row_ptr, col_idx  the CSR (nb = ceil(S / block) rows), on the device.
 *   block    32, 64 or 128: the token block of the CSR.  The kernel works in 64-token key steps:
 *            a 128-token key block is walked as two, two 32-token key blocks share one with a
 *            mask per (32-row query block, 32-key half); every token's allowed key set is the
 *            one the CSR defines at its own block.
 *
 * S need not be a multiple of the block: rows q >= S of a partial last block are neither
 * computed into O nor into lse, and keys k >= S are never weighed.
 * Limits: block in {32, 64, 128}, D in {64, 128}, B*H <= 65535, B*H*S < 2^31.
 * Errors: INVALID_ARGUMENT, UNSUPPORTED (block or D), NOT_DEVICE_POINTER, DEVICE_MISMATCH,
 * CUDA.  Device-side: BAD_SCHEDULE (a row is truncated at its first bad entry), TIMEOUT.
 */
tsa_status tsa_scheduled_attention(const void *Q, const void *K, const void *V,
                                   const int32_t *row_ptr, const int32_t *col_idx, void *O,
                                   tsa_dtype dtype, int64_t B, int64_t H, int64_t S, int64_t D,
                                   int64_t block, float scale, tsa_stream_t stream);

/*
 * tsa_scheduled_attention that also writes, for every query row, the log-sum-exp of its scaled
 * scores over the allowed keys: lse[l][q] = log(sum_{k allowed} exp(scale * <Q[l][q], K[l][k]>))
 * (natural log; -inf for a row without keys).  The backward pass recomputes P from it.
 *
 *   lse  out, [B*H, S] float32 device array, 4-byte aligned (16-byte for the backward call),
 *        or NULL (then this is tsa_scheduled_attention).
 * Arguments, limits and errors otherwise as tsa_scheduled_attention.
 */
tsa_status tsa_scheduled_attention_fwd(const void *Q, const void *K, const void *V,
                                       const int32_t *row_ptr, const int32_t *col_idx, void *O,
                                       float *lse, tsa_dtype dtype, int64_t B, int64_t H, int64_t S,
                                       int64_t D, int64_t block, float scale, tsa_stream_t stream);

/*
 * Backward pass of the scheduled attention (the mirror page's segment-boundary record notes
 * that the merged kernel has none; this is the chain rule of the forward above).  With P the
 * softmax of the scaled scores over each query's allowed keys and dO the upstream gradient:
 *   Delta_q = <dO_q, O_q>,  dS = P o (dO V^T - Delta),
 *   dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q
 * per lane, fp32 accumulation from the 16-bit inputs, results rounded to the input dtype.  P is
 * recomputed from `lse` as written by tsa_scheduled_attention_fwd for the same inputs and CSR.
 *
 *   Q, K, V, O, dO  in,  [B*H, S, D] of `dtype`, 16-byte aligned; O is the forward's output.
 *   lse             in,  [B*H, S] float32 from tsa_scheduled_attention_fwd, 16-byte aligned.
 *   row_ptr, col_idx the CSR the forward ran with; nnz_cap >= its nnz (row_ptr[nb]), e.g. the
 *                   length of col_idx.
 *   dQ, dK, dV      out, [B*H, S, D] of `dtype`, 16-byte aligned, overlapping no input and no
 *                   other output.
 *   workspace       >= tsa_attention_backward_workspace_bytes(B*H, S, block, nnz_cap) bytes,
 *                   256-byte aligned (Delta per row, the transposed schedule and its bitmap of
 *                   nb^2 bits); its contents on entry do not matter.
 *
 * Limits: block in {64, 128} (a CSR of 128-token blocks is first expanded on the GPU into the
 * 64-token CSR with the same allowed keys: rows 2p and 2p+1 hold 64-blocks 2j and 2j+1 of each
 * j < p, plus 2p, and 2p+1 for row 2p+1, when p is in row p; a 32-token CSR is UNSUPPORTED),
 * D in {64, 128}, ceil(S/64) <= 8192 (a partial last block is allowed: its rows are stored one
 * by one, never past the lane's last row), B*H <= 65535,
 * B*H*S < 2^31.  Errors: INVALID_ARGUMENT, UNSUPPORTED, CAPACITY (workspace), NOT_DEVICE_POINTER,
 * DEVICE_MISMATCH, CUDA.  Device-side: BAD_SCHEDULE (a row is cut at its first bad entry, as in
 * the forward), TSA_ERR_DEVICE (nnz above nnz_cap: dK and dV then come out zero), TIMEOUT.
 */
size_t tsa_attention_backward_workspace_bytes(int64_t lanes, int64_t S, int64_t block,
                                              int64_t nnz_cap);
tsa_status tsa_scheduled_attention_backward(const void *Q, const void *K, const void *V,
                                            const void *O, const void *dO, const float *lse,
                                            const int32_t *row_ptr, const int32_t *col_idx,
                                            int64_t nnz_cap, void *dQ, void *dK, void *dV,
                                            tsa_dtype dtype, int64_t B, int64_t H, int64_t S,
                                            int64_t D, int64_t block, float scale, void *workspace,
                                            size_t workspace_bytes, tsa_stream_t stream);

/* Size of the device array behind tsa_build_schedule_noalloc: 16 MiB on every device that
 * loads the library, held until the process exits. */
#define TSA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * tsa_build_schedule for callers that cannot allocate device memory.  Some callers own no
 * device allocator: a plugin running inside a host application that has already reserved the
 * device memory for its own pool, or a latency-bound loop in which cudaMalloc's implicit
 * device-wide synchronization is not acceptable.  This entry point takes no workspace; it
 * uses a fixed scratch array of TSA_NOALLOC_SCRATCH_BYTES inside the library instead and
 * calls no cudaMalloc, cudaFree or other allocating routine.  One caveat for the first call
 * on a device: it looks up the array's device address, and with lazy module loading (the
 * CUDA runtime's default) that lookup may load this library's module on the device and
 * reserve the array's memory right then, which can synchronize the device.  Make that first
 * call outside any latency-critical region and before any stream capture; later calls do
 * neither.  The paper has no counterpart: this is a packaging choice of
 * this library, not part of the method.
 *
 * Arguments, results and limits are those of tsa_build_schedule without `workspace` and
 * `workspace_bytes`.  The scratch needed is tsa_build_schedule_workspace_bytes(lanes, S, D,
 * block); above TSA_NOALLOC_SCRATCH_BYTES the call returns TSA_ERR_CAPACITY without launching
 * anything (for example 64 lanes of [32768, 128] keys need about 35 MiB and are rejected,
 * 64 lanes of [8192, 64] need about 4.2 MiB and fit).
 *
 * The first call on each device looks up the scratch array's device address (with that
 * device current) and caches it (see above).  All calls
 * on a device share the one array: calls that can overlap on the GPU (on different streams
 * without ordering between them) race on it and must be serialized by the caller.  Nothing
 * in the array needs to start at zero; a call never reads what an earlier call left there.
 */
tsa_status tsa_build_schedule_noalloc(const void *K, tsa_dtype dtype, int64_t lanes, int64_t S,
                                      int64_t D, int64_t block, int64_t sink,
                                      int64_t local_radius, int64_t topk, int32_t *row_ptr,
                                      int32_t *col_idx, int64_t col_cap, double *salience_sq,
                                      tsa_stream_t stream);

/*
 * One forward step of the path from HOST memory: the topology schedule built from K, the
 * scheduled attention over it, and O back in host memory -- the calls above, with the
 * host<->device copies overlapped with the work.  Lanes go in chunks of `lane_chunk` (0: a
 * sixteenth of the lanes): the K chunks are copied first and each one's block sums run as soon
 * as it lands, then the schedule; the Q and V chunks follow, each chunk's attention starts
 * when its Q and V have landed, and its O is copied back on a third stream while the next
 * chunk runs.  The copies use two streams and a set of events of the library's own, created by
 * the first call on each device and kept until the process exits (calls on one device from
 * several host threads take turns enqueueing); the work runs on `stream`, and `stream`
 * continues only after every copy has been made (the call is asynchronous like the others:
 * synchronize `stream` before reading hO).
 *
 *   hQ, hK, hV   in, [B*H, S, D] of `dtype` in host memory (page-locked for the copies to run
 *                asynchronously and overlap; pageable memory works, slower)
 *   hO           out, host memory of the same shape
 *   dQ, dK, dV, dO   device buffers of the same size, 16-byte aligned, not overlapping: the
 *                device copies of the inputs and the device output (left valid after the call)
 *   row_ptr, col_idx, col_cap, workspace, workspace_bytes, block, sink, local_radius, topk,
 *                tie_break: as tsa_build_schedule_ex (workspace >=
 *                tsa_build_schedule_workspace_bytes(B*H, S, D, block)); the schedule stays in
 *                row_ptr / col_idx
 *   scale        as tsa_scheduled_attention
 *
 * Limits: those of tsa_build_schedule_ex and tsa_scheduled_attention; at most 4096 chunks.
 * Errors: INVALID_ARGUMENT (also for a device or managed pointer given as host memory),
 * UNSUPPORTED, CAPACITY, NOT_DEVICE_POINTER, DEVICE_MISMATCH, CUDA.
 */
tsa_status tsa_topology_attention_host(const void *hQ, const void *hK, const void *hV, void *hO,
                                       tsa_dtype dtype, int64_t B, int64_t H, int64_t S, int64_t D,
                                       int64_t block, int64_t sink, int64_t local_radius, int64_t topk,
                                       tsa_tie_break tie_break, float scale, void *dQ, void *dK, void *dV,
                                       void *dO, int32_t *row_ptr, int32_t *col_idx, int64_t col_cap,
                                       void *workspace, size_t workspace_bytes, int64_t lane_chunk,
                                       tsa_stream_t stream);

/*
 * Synchronizes `stream`, then returns and clears the device status word of the current
 * device: TSA_OK, or the first of TIMEOUT, BAD_SCHEDULE, CAPACITY-on-device (reported as
 * TSA_ERR_DEVICE) raised by any call since the last read.  TSA_ERR_CUDA if the
 * synchronization itself fails.
 */
tsa_status tsa_last_device_status(tsa_stream_t stream);

/*
 * Test hook for the failure path (no counterpart on the pages).  With `on` = 1, every later
 * scheduled-attention launch of this process has its first CTA withhold the scores of its
 * first key block, so that CTA's softmax wait runs out after its bound (1 s): the launch
 * gives up cleanly -- no trap, no hang; every CTA drains what it issued and frees its
 * tensor memory -- and tsa_last_device_status() then reports TSA_ERR_TIMEOUT.  The output of
 * such a launch is unspecified.  `on` = 0 restores normal launches (the default); the CUDA
 * context stays usable throughout.  Process-wide, not thread-safe against concurrent
 * launches, and meant for tests only.  TSA_ERR_INVALID_ARGUMENT for other values.
 */
tsa_status tsa_debug_set_wait_injection(int on);

#ifdef __cplusplus
}
#endif

#endif /* TSA_H_ */
