/*
 * pw.h -- C ABI of libpw, the GB300 (sm_103a) library for the data-parallel hot
 * path of PagedWeight's fused mixed-precision Any-Precision MoE expert layer.
 *
 * Source of every operation: "PagedWeight: Efficient MoE LLM Serving with
 * Dynamic Quality-Aware Weight Quantization" (arXiv text).  Section, equation
 * and figure are cited beside each call.
 *
 * Conventions
 *  - Every call returns int: PW_OK (0) or a negative PW_ERR_* code; the
 *    message of the last failure on the calling thread is pw_last_error().
 *    No C++ exception crosses this boundary.
 *  - Arguments are validated on the host before anything is enqueued.
 *  - Device memory is always caller-owned.  libpw never allocates or frees
 *    device memory; scratch space is a caller-provided workspace.
 *  - "stream" is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Device work is enqueued on it and the call returns without
 *    synchronising.  Pointers named d_* are device pointers; h_* are host.
 *  - fp16 data is IEEE binary16 passed as uint16_t.
 *  - Failures that only the device can see (a wait that ran out, a block that
 *    is routed to but not committed) are written to a caller-provided int32
 *    status word in device memory (d_status) with the PW_ERR_* code; the
 *    caller reads it after synchronising.  The kernels never trap.
 *  - The page table is host state and is not thread-safe.
 */
#ifndef PW_H_
#define PW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PW_OK 0
#define PW_ERR_INVALID_ARG (-1)
#define PW_ERR_UNSUPPORTED (-2)   /* bitwidth or shape this library does not handle */
#define PW_ERR_NOT_RESIDENT (-3)  /* a page needed for the requested bitwidth is not attached */
#define PW_ERR_CUDA (-4)          /* a CUDA runtime call failed; see pw_last_error() */
#define PW_ERR_TIMEOUT (-5)       /* a bounded in-kernel wait ran out (device status only) */
#define PW_ERR_WORKSPACE (-6)     /* workspace too small or misaligned */
#define PW_ERR_BUSY (-7)          /* a transfer of this page is still in flight */

#define PW_MAX_BITS 8
#define PW_LAYOUT_TILED 1

/* Message describing the last failure on this thread ("" if none). */
const char* pw_last_error(void);

/* ------------------------------------------------------------------------ */
/* Bit-plane packer (§1 and Figure 3: the overlaid bit-plane format)          */
/* ------------------------------------------------------------------------ */

/* Bytes of one bit-plane of a rows x cols block in `layout` (= rows*cols/8).
 * Returns 0 if the shape is not supported: the tiled layout needs
 * rows % 128 == 0 and cols % 128 == 0. */
size_t pw_plane_bytes(int64_t rows, int64_t cols, int layout);

/* Split parent-bit indices into bit-planes.
 *  d_idx       device uint8 [rows][cols], row-major, every value < 2^parent_bits
 *  parent_bits P in 1..8
 *  h_planes    HOST array of P device pointers, each to pw_plane_bytes() bytes,
 *              16-byte aligned; plane 0 receives the most significant bit, so
 *              the top b planes hold the b-bit index idx >> (P - b)
 *  layout      PW_LAYOUT_TILED (the only layout), defined element by element:
 *                half = n / (rows/2), r = n % (rows/2), strip = r / 64, rr = r % 64
 *                pos = 32*(rr/16) + rr%16 + 16*half
 *                tile = j / 128, jj = j % 128, t = jj % 32
 *                bit (n, j) is bit 4*(t%8) + t/8 of the little-endian uint32
 *                at byte (strip*(cols/128) + tile)*2048 + 16*pos + 4*(jj/32)
 *              i.e. 2048-byte tiles of a 128-row strip x 128 columns,
 *              strip-major; row position pos owns 16 bytes of each tile, and
 *              positions pos and pos+16 of a warp hold rows m and rows/2+m
 *              (the gate and up rows of a gate_up block).
 * Values >= 2^P are masked to their low P bits.  Asynchronous on `stream`. */
int pw_pack_bitplanes(const uint8_t* d_idx, int64_t rows, int64_t cols, int parent_bits,
                      uint32_t* const* h_planes, int layout, void* stream);

/* Rearrange a LUT (fp16 [rows][2^bits] row-major, one row of centroids per
 * output row, Figure 3 caption) into the tiled LUT layout that LUT pages are
 * stored in (pw_page_table_attach_lut):
 *   with half, strip, rr of row n as above, w = rr/16, i = rr%16 + 16*half,
 *   entry c of row n is the fp16 at byte
 *     (strip*2^bits + c)*256 + 4*((w%2)*32 + i) + 2*(w/2)
 * so the table of a 128-row strip is one contiguous run of 2^bits*256 bytes
 * (the order of the kernels' shared LUT region; a unit copies it in one
 * piece).  d_out: rows*2^bits*2 bytes, 16-byte aligned, not d_lut.
 * rows % 128 == 0, bits 1..8.  Asynchronous on `stream`. */
int pw_pack_lut(const uint16_t* d_lut, int64_t rows, int bits, uint16_t* d_out, void* stream);

/* ------------------------------------------------------------------------ */
/* Weight page table (§3 and §3.1; Eq. 3)                                      */
/* ------------------------------------------------------------------------ */

/* Shape and supported bitwidths B_i = {seed_bits .. parent_bits} of one
 * per-expert linear-block i = (layer, expert, gate_up|down). */
typedef struct pw_block_info {
  int64_t rows;      /* output rows N (gate_up: 2I, down: H) */
  int64_t cols;      /* input columns K (gate_up: H, down: I) */
  int32_t parent_bits;
  int32_t seed_bits;
  int32_t layout;    /* PW_LAYOUT_TILED */
  int32_t reserved;
} pw_block_info;

typedef struct pw_page_table pw_page_table;

/* Bytes of the device descriptor array for n_blocks blocks (see _sync). */
size_t pw_desc_bytes(int n_blocks);

/* Create a table of n_blocks rows.  Block ids are chosen by the caller; the
 * fused layer reads block (layer*E + e)*2 + u, u = 0 gate_up, 1 down.
 * Every block starts uncommitted (q = 0, d = 0) with no pages attached. */
int pw_page_table_create(pw_page_table** out, int n_blocks, const pw_block_info* h_info);
int pw_page_table_destroy(pw_page_table* t);

/* Attach (borrow) the device buffer of bit-plane `plane` (0 = MSB) of a block;
 * marks that plane GPU-resident.  The buffer must stay valid while attached. */
int pw_page_table_attach_plane(pw_page_table* t, int block, int plane, const uint32_t* d_plane);

/* Attach the LUT of bitwidth `bits` (seed..parent): rows*2^bits fp16 in the
 * tiled LUT layout (pw_pack_lut), 16-byte aligned, one row of centroids per
 * output row (Figure 3 caption). */
int pw_page_table_attach_lut(pw_page_table* t, int block, int bits, const uint16_t* d_lut);

/* Record the planner's desired bitwidth d_i (bookkeeping; §3: q_i, not d_i,
 * is what inference uses).  d must be in B_i. */
int pw_page_table_set_desired(pw_page_table* t, int block, int d);

/* Commit q_i = q (§3.1 and §3.3 ordering rules).
 *  Lowering (q < q_i): commits q at once; planes q..P-1 and LUTs q+1..P become
 *  unreferenced, are detached, and are reported in *released_mask (bit p for
 *  plane p, bit 8+b for the LUT of bitwidth b) so the caller can free them
 *  once the stream has passed every launch that used them -- except pages
 *  whose offload copy is still in flight, which stay attached until
 *  pw_page_table_poll sees the copy finish (see pw_page_offload).  The planes
 *  below q are not touched.
 *  Raising (q > q_i): only allowed once planes 0..q-1 and the LUTs seed..q are
 *  attached (reload first, then raise); otherwise PW_ERR_NOT_RESIDENT and
 *  nothing changes.  q must be in B_i.  released_mask may be NULL. */
int pw_page_table_set_bits(pw_page_table* t, int block, int q, uint64_t* released_mask);

/* Committed q_i, desired d_i and the attached-page mask (bit p plane p,
 * bit 8+b LUT b) of a block; any out pointer may be NULL. */
int pw_page_table_get(const pw_page_table* t, int block, int* q, int* d, uint64_t* resident_mask);

/* M_i^b of Eq. 3: bytes block i holds on the GPU at bitwidth b -- b planes of
 * rows*cols/8 bytes plus the fp16 LUTs of every bitwidth seed..b.  Returns -1
 * for an invalid block or b outside B_i. */
int64_t pw_page_table_bytes(const pw_page_table* t, int block, int b);

/* Sum over blocks of M_i^{q_i} (uncommitted blocks count 0). */
int64_t pw_page_table_resident_bytes(const pw_page_table* t);

/* Upload the descriptors of all blocks (committed q, plane and LUT_q
 * pointers, shape) to d_desc (pw_desc_bytes(n_blocks) bytes, 16-byte aligned)
 * with an asynchronous copy on `stream`.  The fused kernels read only this
 * array, so a commit becomes visible to launches enqueued after the sync. */
int pw_page_table_sync(pw_page_table* t, void* d_desc, size_t desc_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Asynchronous page movement (§3.1 page states; §3.3 and Figure 4)          */
/* ------------------------------------------------------------------------ */
/* A weight page is one bit-plane or the LUT of one bitwidth of a block.  Page
 * ids: plane p (0 = MSB) is page p; the LUT of bitwidth b is page 8 + b.  A
 * page is GPU-resident (attached), may also hold a complete host copy
 * (CPU-resident), and may be in transfer.  Transfers are one cudaMemcpyAsync
 * each on the caller's copy stream (normally not the compute stream, so the
 * copies overlap the fused layer), tracked by an event the table owns; the
 * table notices that a transfer finished only in pw_page_table_poll.
 *
 * Offload (§3.3): pw_page_offload copies a GPU-resident page to host memory;
 * the caller then lowers q_i with pw_page_table_set_bits, which retires pages
 * above q_i at once unless their offload copy is still in flight -- those
 * stay attached until the poll that sees the copy finish detaches them and
 * reports them through pw_page_table_take_released.  Reload (§3.1 ordering):
 * pw_page_reload copies the host copy into a caller device buffer; the page
 * is attached only by the poll that sees the copy finish, so raising q_i
 * before then fails with PW_ERR_NOT_RESIDENT.  Buffers stay caller-owned; the
 * host buffers should be pinned for the copies to run asynchronously. */
#define PW_PAGE_LUT(b) (8 + (b))
#define PW_PAGE_GPU 1      /* attached: usable by the kernels when committed */
#define PW_PAGE_CPU 2      /* a complete host copy exists */
#define PW_PAGE_TO_CPU 4   /* offload copy in flight */
#define PW_PAGE_TO_GPU 8   /* reload copy in flight */

/* Bytes of a page (rows*cols/8 for a plane, rows*2^b*2 for LUT b); -1 if the
 * block or page does not exist. */
int64_t pw_page_bytes(const pw_page_table* t, int block, int page);

/* Start copying a GPU-resident page to h_dst (pw_page_bytes bytes) on
 * copy_stream.  PW_ERR_NOT_RESIDENT if the page is not attached, PW_ERR_BUSY
 * if a transfer of it is in flight.  The copy reads the attached buffer, so
 * the caller orders copy_stream after whatever wrote it. */
int pw_page_offload(pw_page_table* t, int block, int page, void* h_dst, void* copy_stream);

/* Start copying a page from host memory (h_src, or when h_src is NULL the
 * page's own completed host copy) into d_dst (16-byte aligned, pw_page_bytes
 * bytes) on copy_stream.  The page must not be attached (PW_ERR_INVALID_ARG)
 * and must have no transfer in flight (PW_ERR_BUSY); PW_ERR_NOT_RESIDENT if
 * h_src is NULL and no host copy exists. */
int pw_page_reload(pw_page_table* t, int block, int page, const void* h_src, void* d_dst, void* copy_stream);

/* Advance every finished transfer: an offload marks the host copy complete
 * and detaches the page if it is above q_i; a reload attaches its buffer.
 * *in_flight (may be NULL) gets the number of transfers still running.
 * Host only: never waits. */
int pw_page_table_poll(pw_page_table* t, int* in_flight);

/* Pages of a block that a poll detached after their offload copy finished
 * (bit p plane p, bit 8+b LUT b), cleared by the call; the caller frees those
 * device buffers once the compute stream is past the launches that used
 * them. */
int pw_page_table_take_released(pw_page_table* t, int block, uint64_t* released_mask);

/* State bits (PW_PAGE_*) of a page, its attached device buffer and its host
 * buffer; any out pointer may be NULL. */
int pw_page_state(const pw_page_table* t, int block, int page, int* state, const void** d_ptr, void** h_ptr);

/* ------------------------------------------------------------------------ */
/* Routing (§2.1: top-K experts per token; Eq. 1: routing mass)                */
/* ------------------------------------------------------------------------ */

/* Top-k routing of fp32 logits [T][E] (finite values), one launch:
 *  d_ids     int32 [T][k]   chosen experts by decreasing logit, ties to the
 *                           lower expert index
 *  d_w       fp32  [T][k]   softmax probabilities renormalised over the k picks
 *  d_offsets int32 [E+1]    offsets[e] = first position of expert e
 *  d_perm    int32 [T*k]    perm[pos] = slot t*k+j, positions ordered by
 *                           (expert, token, j)
 *  d_inv_perm int32 [T*k]   inverse of perm
 *  d_mass_accum fp32 [E] or NULL: adds sum_t sum_j w[t][j]*[ids[t][j] == e]
 *                           (the numerator of Eq. 1; the denominator is T)
 * Limits: 1 <= k <= E <= 256, k <= 16, 0 <= T <= 2^20.  T = 0 writes the
 * offsets (all zero) and nothing else. */
int pw_moe_route_topk(const float* d_logits, int T, int E, int k, int32_t* d_ids, float* d_w,
                      int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm,
                      float* d_mass_accum, void* stream);

/* Routing with S shared experts (Table 1: Qwen1.5-MoE-A2.7B has 60 routed
 * plus 4 shared experts, Gemma-4-26B-A4B 128 plus 1): experts every token
 * passes through, added to the routed output.  The pages give no gate for
 * them; here each has weight 1.  Every token gets K = k + S slots: its top-k
 * routed experts (as pw_moe_route_topk over the E routed logits) followed by
 * the shared experts E .. E+S-1 with w = 1.  Outputs are over E + S experts
 * and K slots: ids and w [T][K], offsets [E+S+1], perm and inv_perm [T*K],
 * mass [E+S] (shared experts receive T per call); the permutation stays
 * stable by (expert, token, slot).  pw_moe_apl_ffn then runs with E + S
 * experts and K for k.  Limits: 1 <= k <= E, S >= 0, E + S <= 256,
 * k + S <= 16. */
int pw_moe_route_topk_shared(const float* d_logits, int T, int E, int k, int S, int32_t* d_ids,
                             float* d_w, int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm,
                             float* d_mass_accum, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused mixed-precision MoE expert layer (§3.3, "Fused Mixed-Precision MoE Kernel") */
/* ------------------------------------------------------------------------ */

/* Workspace bytes pw_moe_apl_ffn needs for this problem size. */
size_t pw_moe_apl_ffn_workspace(int T, int H, int I, int E, int k);

/* One launch computing, for every token t,
 *   y[t] = sum_j w[t][j] * down_e( silu(gate_e x_t) * up_e x_t ),  e = ids[t][j]
 * where each expert's gate_up (rows [0,I) gate, [I,2I) up) and down blocks
 * are read at their own committed bitwidth q_i straight from the bit-planes:
 * only the top q_i planes are loaded, the q_i-bit index is looked up in that
 * block's LUT_{q_i} (fp16), products accumulate in fp32, the activation h is
 * rounded to fp16, and y is rounded to fp16.  Experts with no tokens are not
 * read.  Blocks of expert e in `layer` are descriptor entries
 * (layer*E + e)*2 + {0: gate_up, 1: down} of d_desc (see _sync).
 *  d_x  fp16 [T][H], 16-byte aligned;  d_y fp16 [T][H] (written), 8-byte
 *  aligned;  routing arrays as produced by
 *  pw_moe_route_topk (d_ids may be NULL: it is not read);
 *  d_ws workspace of pw_moe_apl_ffn_workspace() bytes, 256-byte aligned,
 *  contents need not be initialised;
 *  d_status int32, set to a PW_ERR_* code on a device-side failure (left
 *  untouched on success, so the caller zeroes it beforehand).
 * Shapes: H % 128 == 0, I % 128 == 0, committed bitwidths 2..8.
 * The call picks the token-tile width from the average number of tokens per
 * expert (T*k/E): tiles of 16 tokens below 12, else of 64; and the path:
 * below 48 the decode path (down projection split over I in 3072-column
 * parts), else the prefill path (no split).  The top-k weighted combine runs
 * over the whole grid after the last unit.  All run on the tcgen05 tensor cores;
 * pw_moe_apl_ffn_ex can force either path. */
int pw_moe_apl_ffn(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I,
                   int E, int k, const int32_t* d_ids, const float* d_w,
                   const int32_t* d_offsets, const int32_t* d_perm, const int32_t* d_inv_perm,
                   void* d_ws, size_t ws_bytes, uint16_t* d_y, int32_t* d_status, void* stream);

/* Same computation as pw_moe_apl_ffn, for callers that cannot allocate
 * device memory: code running while a CUDA graph is being captured, plugin
 * hosts whose memory contract forbids allocation during inference, and
 * real-time loops where an allocation's latency or failure is not acceptable.
 * The paper has no counterpart; this is an interface convenience.
 *
 * The scratch space lives in a fixed array inside libpw of
 * PW_NOALLOC_SCRATCH_BYTES (32 MiB), which every GPU that loads the library
 * holds until the process exits.  A call is accepted when the workspace of
 * the path it takes fits the array, else it fails with PW_ERR_WORKSPACE
 * before anything is enqueued.  The decode path (below 48 assignments per
 * expert on average) needs more workspace per token than the prefill path,
 * so the accepted token counts are not one interval: for the Mixtral-8x7B
 * shape at top-2 they are T <= 141 (decode path) and 192 <= T <= 315
 * (prefill path).  pw_moe_apl_ffn_workspace returns the larger of the two
 * paths' sizes, so workspace(T) <= PW_NOALLOC_SCRATCH_BYTES is a sufficient
 * (not a necessary) check.  This entry point allocates nothing itself (no
 * cudaMalloc/cudaFree, no allocating library routine).
 *  - The first call on a device looks up the array's device address (a one-off
 *    set-up, once per device, with that device current); make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after cudaDeviceReset on a device it is stale, and this entry
 *    point must not be called on that device again.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls that overlap on the GPU (different streams without ordering, or
 *    concurrent host threads) race and give wrong results.  Serialise them.
 * Arguments, layouts and errors are those of pw_moe_apl_ffn. */
#define PW_NOALLOC_SCRATCH_BYTES (32u << 20)
int pw_moe_apl_ffn_noalloc(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I,
                           int E, int k, const int32_t* d_ids, const float* d_w,
                           const int32_t* d_offsets, const int32_t* d_perm,
                           const int32_t* d_inv_perm, uint16_t* d_y, int32_t* d_status,
                           void* stream);

/* Options of pw_moe_apl_ffn_ex (zero-initialise, then set what you need). */
#define PW_PATH_AUTO 0
#define PW_PATH_DECODE 1   /* down split over I; routing inside the routed call's launch */
#define PW_PATH_PREFILL 2  /* down over all of I; routing as its own launch in a routed call */
#define PW_FFN_FLAG_TEST_DROP_ONE_ARRIVAL 1u  /* test hook: one gate_up unit never
                                                 signals completion, so the waits
                                                 that depend on it run out */
#define PW_FFN_FLAG_STRIP_COMBINE 2u          /* the CTA that finishes a 128-row
                                                 strip's last down unit combines
                                                 that strip, instead of the whole
                                                 grid combining after the last
                                                 unit (same result, bit for bit) */
/* Which units multiply the dequantised weights with the tokens:
 *  PW_KERNEL_AUTO         the library's choice (the tensor cores: measured
 *                         faster at every batch size, see below);
 *  PW_KERNEL_TENSOR       tcgen05 MMAs on 16-, 64- or 128-token tiles;
 *  PW_KERNEL_CUDA_CORES   fp32 FMAs in the dequantising warps on 2-token
 *                         tiles (a split-K GEMV: every unit sums its rows
 *                         over its K range per set of warps; meant for one or
 *                         two tokens per expert, correct for any batch).
 * Results agree within the output tolerance, not bit for bit (the two sum
 * the products in different orders). */
#define PW_KERNEL_AUTO 0
#define PW_KERNEL_TENSOR 1
#define PW_KERNEL_CUDA_CORES 2
typedef struct pw_ffn_options {
  int32_t path;              /* PW_PATH_* */
  uint32_t flags;            /* PW_FFN_FLAG_* */
  uint32_t wait_timeout_us;  /* bound of each in-kernel wait; 0 = 2 s */
  int32_t shared_experts;    /* routed call only: S shared experts (see pw_moe_route_topk_shared) */
  int32_t kernel;            /* PW_KERNEL_* */
  int32_t reserved[3];
} pw_ffn_options;

int pw_moe_apl_ffn_ex(const void* d_desc, int layer, const uint16_t* d_x, int T, int H, int I,
                      int E, int k, const int32_t* d_ids, const float* d_w,
                      const int32_t* d_offsets, const int32_t* d_perm, const int32_t* d_inv_perm,
                      void* d_ws, size_t ws_bytes, uint16_t* d_y, int32_t* d_status,
                      const pw_ffn_options* opts, void* stream);

/* Routing and the fused expert layer in one launch (§3.3: routing belongs to
 * the fused kernel together with the experts' work and the weighted sum).
 * Computes what pw_moe_route_topk followed by pw_moe_apl_ffn computes, with
 * the same results bit for bit:
 *  d_logits fp32 [T][E] router logits (input, finite values);
 *  d_ids, d_w, d_offsets, d_perm, d_inv_perm: the routing arrays, OUTPUTS
 *    here (layouts as in pw_moe_route_topk), none may be NULL when T > 0;
 *  d_mass_accum fp32 [E] or NULL: the routing mass is added as in
 *    pw_moe_route_topk.
 * Batches one warp routes (at most 32 tokens, 8 experts and 4 slots per
 * token, shared experts included) on the decode path (T*k < 48*E) are routed
 * by one warp of the fused kernel at the start of the launch while the other
 * CTAs wait for it (bounded; a timeout sets d_status to PW_ERR_TIMEOUT).
 * Other batches are routed by a routing launch that runs first on the same
 * stream.
 * T = 0 writes the offsets (all zero) and nothing else (d_logits may then be
 * NULL).  E and k count the routed experts (the logits' width and top-k);
 * with options->shared_experts = S (the _ex form) routing is that of
 * pw_moe_route_topk_shared and the layer runs over E + S experts (descriptor
 * entries of the layer: E + S experts) and k + S slots, so the routing arrays
 * are sized for them.  Every other argument, limit and error is that of
 * pw_moe_apl_ffn. */
int pw_moe_route_apl_ffn(const void* d_desc, int layer, const uint16_t* d_x, const float* d_logits,
                         int T, int H, int I, int E, int k, int32_t* d_ids, float* d_w,
                         int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm,
                         float* d_mass_accum, void* d_ws, size_t ws_bytes, uint16_t* d_y,
                         int32_t* d_status, void* stream);
int pw_moe_route_apl_ffn_ex(const void* d_desc, int layer, const uint16_t* d_x, const float* d_logits,
                            int T, int H, int I, int E, int k, int32_t* d_ids, float* d_w,
                            int32_t* d_offsets, int32_t* d_perm, int32_t* d_inv_perm,
                            float* d_mass_accum, void* d_ws, size_t ws_bytes, uint16_t* d_y,
                            int32_t* d_status, const pw_ffn_options* opts, void* stream);

/* Several independent MoE layers in one fused launch (plus one routing
 * launch before it when the layers' batches are larger than one warp routes,
 * as in pw_moe_route_apl_ffn): the routed call of
 * pw_moe_route_apl_ffn_ex for layers layer0 .. layer0+L-1 of the descriptor
 * array, each with its own T tokens (§3.3's fused kernel, applied to a stack
 * of layers whose inputs are all known, e.g. a decode stack with independent
 * per-layer batches).  The layers run as one layer of L*T tokens and
 * L*(E+S) experts whose routing never crosses layers, so one persistent grid
 * works through every layer's units and the per-launch start-up and tail are
 * paid once.  Layouts, all arrays concatenated layer after layer:
 *  d_x fp16 [L][T][H], d_logits fp32 [L][T][E], d_y fp16 [L][T][H];
 *  d_ids int32 [L][T][k+S] (each layer's own expert ids, 0 .. E+S-1) and
 *  d_w fp32 [L][T][k+S];
 *  d_offsets int32 [L*(E+S)+1], d_perm and d_inv_perm int32 [L*T*(k+S)] in
 *  the concatenated index space: layer l's expert e starts at
 *  d_offsets[l*(E+S)+e], and its assignment slots are l*T*(k+S) + t*(k+S) + j;
 *  d_mass_accum fp32 [L][E+S] or NULL.
 * Workspace: pw_moe_apl_ffn_workspace(L*T, H, I, L*(E+S), k+S).  L*(E+S) must
 * be at most 256.  Every result equals that of L pw_moe_route_apl_ffn_ex
 * calls bit for bit (after the index shift above); every other argument,
 * limit and error is that of pw_moe_route_apl_ffn_ex. */
int pw_moe_route_apl_ffn_layers(const void* d_desc, int layer0, int L, const uint16_t* d_x,
                                const float* d_logits, int T, int H, int I, int E, int k,
                                int32_t* d_ids, float* d_w, int32_t* d_offsets, int32_t* d_perm,
                                int32_t* d_inv_perm, float* d_mass_accum, void* d_ws, size_t ws_bytes,
                                uint16_t* d_y, int32_t* d_status, const pw_ffn_options* opts,
                                void* stream);

/* ------------------------------------------------------------------------ */
/* Test exports: they run the same device dequant code as the fused layer.     */
/* ------------------------------------------------------------------------ */

/* b-bit overlay indices of `block` of the table, read from its top b
 * attached planes: d_idx_out uint8 [rows][cols].  b must be 1..8 and planes
 * 0..b-1 attached (else PW_ERR_NOT_RESIDENT). */
int pw_unpack_indices(const pw_page_table* t, int block, int b, uint8_t* d_idx_out,
                      void* stream);

/* out[m][n] = sum_j W[n][j] * x[m][j], W = LUT_q[n][idx_q[n][j]] of `block`
 * at its committed bitwidth q (2..8): d_x fp16 [M][cols], d_out fp32
 * [M][rows], fp32 accumulation.  M >= 0; M <= 2 runs on the CUDA-core
 * instance of the fused kernel, larger M on its tensor-core instances.  Its work-ticket counter is one
 * array inside the library, zeroed by each call: calls that overlap on the
 * GPU (different streams without ordering) race.  Serialise them. */
int pw_apl_linear(const pw_page_table* t, int block, const uint16_t* d_x, int M,
                  float* d_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PW_H_ */
