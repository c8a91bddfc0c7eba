/*
 * cce.h -- C ABI of the GB300 (sm_103a) Cut Cross-Entropy library.
 *
 * The operation is the classifier-head matmul fused with cross-entropy over a
 * large vocabulary, computed forward and backward without ever writing the
 * N x V logit matrix to device memory:
 *
 *   loss_i = LSE_i - C[x_i] . E_i,   LSE_i = log sum_v exp(C_v . E_i)
 *
 * ("Cut Your Losses in Large-Vocabulary Language Models", section "The
 * Mathematical Decomposition"; "Cut Cross-Entropy: Training Loss Without the
 * Logit Matrix ...", section "The decomposition").  The backward pass
 * recomputes the logits tile by tile, forms G = softmax - onehot(x) and
 * contracts it into dE = G C and dC = G^T E ("Cut Your Losses ...", sections
 * "Memory-Efficient Linear-Log-Sum-Exp, Backward Pass (Algorithm 3)" and
 * "The Combined Backward Pass (Algorithm 4)"), skipping tiles whose every
 * |G| < filter_eps ("Gradient Filtering").
 *
 * Conventions shared by every call
 * --------------------------------
 * - Layouts: E [N, D] bf16, C [V, D] bf16, dE [N, D] bf16, dC [V, D] bf16,
 *   all row-major and dense (row pitch D elements); x [N] int64; lse [N] fp32.
 *   bf16 buffers are passed as void* (raw 16-bit IEEE bfloat16 values).
 * - Every pointer is a DEVICE pointer of the current CUDA device unless its
 *   comment says host.  The caller owns every buffer, including the
 *   workspace; the library allocates no device memory.
 * - Requirements checked synchronously, before anything is launched:
 *   non-null pointers; 1 <= N, V < 2^31; 1 <= D < 2^31 with D % 8 == 0 (16-byte
 *   row pitch for TMA); E, C, dE, dC, lse, loss and workspace 16-byte aligned;
 *   ws_bytes >= the matching *_workspace_bytes(); a valid reduction; a finite
 *   filter_eps >= 0; current device of compute capability 10.3.  A failed check
 *   returns its status and launches nothing.
 * - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *   stream).  Outputs are overwritten, never accumulated into.
 * - Targets: x_i must lie in [0, V) or equal ignore_index.  Rows with
 *   x_i == ignore_index add no loss and receive exactly zero gradient
 *   ("cut-cross-entropy" kernel card, section "Correctness").  An out-of-range
 *   target does not cause an out-of-bounds access: the row is treated as
 *   ignored and CCE_DEVERR_TARGET_RANGE is OR-ed into *dev_err, which the
 *   caller reads after synchronising (the Python binding raises on it).
 * - Device error word (*dev_err, int32, device memory, optional: NULL allowed):
 *   bits are only ever OR-ed in; the caller zeroes it.
 *     CCE_DEVERR_TARGET_RANGE  a target was outside [0, V) and not ignored
 *     CCE_DEVERR_TIMEOUT       a pipeline wait inside a kernel ran out (a
 *                              bug); the kernel returned early, outputs are
 *                              undefined.
 */
#ifndef CCE_GB300_H
#define CCE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CCE_OK = 0,
  CCE_ERR_NULL = 1,         /* a required pointer is NULL */
  CCE_ERR_SHAPE = 2,        /* N, D or V out of range, or D % 8 != 0 */
  CCE_ERR_ALIGN = 3,        /* a buffer is not 16-byte aligned */
  CCE_ERR_ARG = 4,          /* bad reduction or filter_eps */
  CCE_ERR_WORKSPACE = 5,    /* ws_bytes smaller than the query */
  CCE_ERR_DEVICE = 6,       /* current device is not compute capability 10.3 */
  CCE_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed */
  CCE_ERR_TARGET_RANGE = 8, /* status form of CCE_DEVERR_TARGET_RANGE */
  CCE_ERR_TIMEOUT = 9       /* status form of CCE_DEVERR_TIMEOUT */
} cce_status;

typedef enum { CCE_RED_NONE = 0, CCE_RED_SUM = 1, CCE_RED_MEAN = 2 } cce_reduction;

#define CCE_DEVERR_TARGET_RANGE 1
#define CCE_DEVERR_TIMEOUT 2

/* Default gradient-filter threshold, finfo(bf16).eps / 32 = 2^-12
 * ("Cut Cross-Entropy: Training Loss Without the Logit Matrix ...", section
 * "Gradient filtering: the part that makes it fast"). */
#define CCE_FILTER_EPS_DEFAULT 0.000244140625f

/* Bytes of device workspace cce_forward / cce_backward need for these sizes
 * (0 for invalid sizes).  Pure host arithmetic; needs no GPU. */
size_t cce_forward_workspace_bytes(int64_t N, int64_t D, int64_t V);
size_t cce_backward_workspace_bytes(int64_t N, int64_t D, int64_t V);

/*
 * Forward: linear-log-sum-exp with target capture ("Cut Your Losses ...",
 * "Memory-Efficient Linear-Log-Sum-Exp, Forward Pass (Algorithm 2)" and
 * "Memory-Efficient Indexed Matrix Multiplication (Algorithm 1)"; the
 * running (max, sumexp) fold of the "cut-cross-entropy" card's "Method").
 *
 *   E, C, x       inputs as above.
 *   ignore_index  target value of rows to ignore (PyTorch's default is -100).
 *   reduction     CCE_RED_NONE: loss[i] = loss_i for all N rows (0 on ignored
 *                 rows); CCE_RED_SUM: loss[0] = sum_i loss_i;
 *                 CCE_RED_MEAN: loss[0] = sum_i loss_i / max(count, 1), count =
 *                 number of non-ignored rows.  A fully ignored batch gives
 *                 loss 0 and zero gradients, as the "cut-cross-entropy" card
 *                 ("Correctness") states; this differs from PyTorch's
 *                 cross_entropy, whose mean over no rows is NaN.
 *   loss          [N] fp32 for NONE, else [1] fp32 (written).
 *   lse           [N] fp32 (written): LSE_i for every row, ignored rows too.
 *                 Keep it for cce_backward.
 *   workspace     >= cce_forward_workspace_bytes(N, D, V) bytes, scratch.
 *   dev_err       optional device error word (see above).
 * The result is deterministic: repeated calls give bitwise identical outputs.
 */
cce_status cce_forward(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                       int64_t ignore_index, int reduction, float* loss, float* lse, void* workspace,
                       size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * Backward: recompute + G + filter + dE/dC ("Cut Your Losses ...",
 * "The Combined Backward Pass (Algorithm 4)", "Gradient Filtering").
 *
 *   lse           [N] fp32 from cce_forward on the same E, C.
 *   grad_out      device fp32: [1] (SUM, MEAN: the gradient of the reduced
 *                 loss) or [N] (NONE: the gradient of each row's loss).
 *   filter_eps    skip a 128x128 (token x vocab) tile when every unscaled
 *                 |G| = |softmax - onehot| in it is < filter_eps (an entry
 *                 equal to filter_eps keeps the tile); 0 disables the filter.
 *                 Skipped tiles issue no MMA and no store.
 *   dE            [N, D] bf16 (written); ignored rows are exactly +0.
 *   dC            [V, D] bf16 (written, each vocab row by exactly one CTA, no
 *                 atomics); vocab rows whose tiles were all skipped are 0.
 *   workspace     >= cce_backward_workspace_bytes(N, D, V) bytes, scratch.
 *   dev_stats     optional device int64[2] (written): {tiles, skipped tiles}
 *                 over the filter tiles.
 * Rows that take no part (ignored, or with an out-of-range target) are
 * compacted away on the device before the GEMMs ("Cut Your Losses ...",
 * Table A1: removing ignored tokens), so a filter tile is 128 consecutive
 * participating rows x 128 vocabulary entries, and there are
 * ceil(n/128) x ceil(V/128) tiles for n participating rows.
 */
cce_status cce_backward(const void* E, const void* C, const int64_t* x, const float* lse,
                        const float* grad_out, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                        int reduction, float filter_eps, void* dE, void* dC, void* workspace,
                        size_t ws_bytes, int32_t* dev_err, int64_t* dev_stats, void* stream);

/*
 * Forward pass that allocates nothing and takes no workspace.  The pages
 * have no counterpart to this call: it exists for callers that cannot
 * allocate device memory where they need the loss -- code inside a CUDA-graph
 * capture that must not allocate, runtimes whose device memory is entirely
 * owned by their own pool, or hosts that forbid allocation on the hot path.
 * Instead of a caller workspace it uses a scratch array of
 * CCE_NOALLOC_SCRATCH_BYTES that the library declares in device memory; every
 * GPU that loads the library holds that array until the process exits.
 *
 * Arguments, layouts, results and checks are those of cce_forward (it runs
 * the same kernels), minus workspace/ws_bytes.  Returns CCE_ERR_WORKSPACE,
 * launching nothing, when cce_forward_workspace_bytes(N, D, V) exceeds
 * CCE_NOALLOC_SCRATCH_BYTES (16 MiB; query that function to know whether a
 * size fits -- the five benchmark workloads, up to N = 65,536 tokens, need at
 * most 10 MiB).  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture starts.  All calls share the one
 * array: calls whose GPU work overlaps (e.g. on two streams at once) race and
 * must be serialised by the caller.  It never calls cudaMalloc, cudaFree or
 * any allocating routine.
 */
#define CCE_NOALLOC_SCRATCH_BYTES (16u << 20)
cce_status cce_forward_noalloc(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                               int64_t ignore_index, int reduction, float* loss, float* lse, int32_t* dev_err,
                               void* stream);

/*
 * Forward with logit softcapping.  cce_forward is cce_forward_ex with
 * softcap = 0.  With softcap > 0 every logit a becomes softcap * tanh(a /
 * softcap) before the log-sum-exp and the target capture (Gemma 2's final
 * logits; "Cut Your Losses ...", Table A2 times softcapping as a stage of the
 * backward).  softcap must be finite and >= 0, else CCE_ERR_ARG.
 */
cce_status cce_forward_ex(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                          int64_t ignore_index, int reduction, float softcap, float* loss, float* lse,
                          void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * Forward with options.  cce_forward_ex is cce_forward_ex2 with flags = 0.
 * CCE_FWD_SKIP_IGNORED: the rows that take part (target in [0, V) and not
 * ignore_index) are compacted on the device before the GEMM, which then runs
 * over them only ("Cut Your Losses ...", Table A1: removing ignored tokens
 * before the loss); the loss is unchanged, and lse (and loss for
 * CCE_RED_NONE) is 0 on the other rows instead of their LSE.  cce_backward
 * needs only the LSE of rows that take part, so it accepts this lse.  The
 * workspace grows to cce_forward_workspace_bytes_ex(N, D, V, flags) (a compact
 * copy of E: N * D * 2 bytes, plus 24 bytes per row).  Any other flag bit
 * returns CCE_ERR_ARG.
 */
#define CCE_FWD_SKIP_IGNORED 1
size_t cce_forward_workspace_bytes_ex(int64_t N, int64_t D, int64_t V, int flags);
cce_status cce_forward_ex2(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                           int64_t ignore_index, int reduction, float softcap, int flags, float* loss, float* lse,
                           void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * Backward with softcapping and per-output filtering.  cce_backward is
 * cce_backward_ex with softcap = 0 and CCE_FILTER_BOTH.  softcap must match
 * the forward's; the gradient then carries the slope 1 - tanh^2(a / softcap),
 * while the filter still tests |softmax - onehot| before that slope.
 * filter_flags chooses which gradients skip the filtered tiles ("Cut Your
 * Losses ...", "Numerical Stability Variants"):
 *   CCE_FILTER_BOTH  dE and dC skip them (plain CCE);
 *   CCE_FILTER_DE    only dE skips them; dC is computed from every tile, so no
 *                    vocabulary row is starved of gradient (CCE-Kahan-FullC, the
 *                    pages' pretraining setting; accumulation is fp32 here, so
 *                    no Kahan compensation is needed);
 *   CCE_FILTER_DC    only dC skips them (CCE-Kahan-FullE);
 *   0                neither (same as filter_eps = 0).
 * The survival map and dev_stats always describe the filter decisions.
 *
 * CCE_SORT_VOCAB (OR-ed into filter_flags) walks the vocabulary in sorted
 * order ("Cut Your Losses ...", section "Vocabulary Sorting"): tokens are
 * ordered by their logit sum over the rows that take part, ascending, equal
 * sums by token id (the pages sort by the average logit; dividing by the row
 * count does not change the order).  The sums are computed on the device as
 * C_v . (sum of those rows of E) in fp32, in a fixed order, so the order is
 * deterministic.  The filter tiles are then 128 consecutive sorted positions,
 * which groups the tokens that carry softmax mass into few tiles; dE and dC
 * are those of the same gradient (dC in token order: the dC tiles write their
 * token rows directly).  Costs: a pass over C for the sums, a radix sort of V
 * keys, and per vocabulary chunk a gather of its C rows into sorted order;
 * the workspace grows to cce_backward_workspace_bytes_ex(N, D, V, flags).
 * Any other flag bit returns CCE_ERR_ARG.
 */
#define CCE_FILTER_DE 1
#define CCE_FILTER_DC 2
#define CCE_FILTER_BOTH 3
#define CCE_SORT_VOCAB 4
cce_status cce_backward_ex(const void* E, const void* C, const int64_t* x, const float* lse,
                           const float* grad_out, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                           int reduction, float softcap, float filter_eps, int filter_flags, void* dE, void* dC,
                           void* workspace, size_t ws_bytes, int32_t* dev_err, int64_t* dev_stats, void* stream);

/* Workspace of cce_backward_ex for these sizes and flags (0 for invalid
 * sizes or flags).  Equals cce_backward_workspace_bytes() without
 * CCE_SORT_VOCAB; with it, adds the sort keys, the order and its inverse
 * (12 bytes per token), the sort scratch, and one vocabulary chunk of C in
 * sorted order (bf16). */
size_t cce_backward_workspace_bytes_ex(int64_t N, int64_t D, int64_t V, int flags);

/*
 * Backward with a caller-chosen staging budget.  cce_backward_ex is
 * cce_backward_ex2 with max_staging_bytes = 0.  The backward walks the
 * vocabulary in chunks of vc columns ("Cut Your Losses ...", "The Combined
 * Backward Pass (Algorithm 4)", blocked over the vocabulary): per chunk it
 * recomputes the logits, stages the filtered, scaled gradient G-hat of the
 * chunk in the workspace as bf16 [N][vc], and contracts it into dC (the
 * chunk's rows, written once) and into an fp32 dE accumulator [N][D]
 * (stored by the first chunk, added by the later ones).
 * max_staging_bytes bounds that G-hat buffer: vc is the largest multiple of
 * 256 with N * vc * 2 <= max_staging_bytes, at least 256 and at most 65,536
 * (and at most ceil(V / 2) rounded up to 256, so the buffer is never an
 * N x V matrix).  0 selects the default, 512 MiB with vc >= 2048.  A
 * smaller budget lowers the workspace (the other parts are fixed: the fp32
 * dE accumulator, N * D * 4 bytes, and a compact copy of the rows that take
 * part, N * D * 2 bytes) but adds one pass over the dE accumulator (read +
 * write, N * D * 8 bytes) per extra chunk.  Results are the same at every
 * budget up to the fp32 summation order of dE across chunks.  Arguments,
 * checks and status codes otherwise as cce_backward_ex; the workspace must
 * hold cce_backward_workspace_bytes_ex2(N, D, V, flags, max_staging_bytes).
 */
cce_status cce_backward_ex2(const void* E, const void* C, const int64_t* x, const float* lse,
                            const float* grad_out, int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                            int reduction, float softcap, float filter_eps, int filter_flags,
                            size_t max_staging_bytes, void* dE, void* dC, void* workspace, size_t ws_bytes,
                            int32_t* dev_err, int64_t* dev_stats, void* stream);
size_t cce_backward_workspace_bytes_ex2(int64_t N, int64_t D, int64_t V, int flags, size_t max_staging_bytes);
/* The chunk width vc that cce_backward_ex2 uses for N rows, V vocabulary
 * entries and this budget (0 for invalid sizes). */
uint64_t cce_backward_chunk_cols(int64_t N, int64_t V, size_t max_staging_bytes);

/*
 * The two steps of vocabulary sorting, exposed on their own (the backward
 * with CCE_SORT_VOCAB runs the same kernels on its compacted rows).
 *
 * cce_vocab_logit_sums: sums[v] (fp32, [V], written) = sum over the rows i
 *   that take part (x_i in [0, V) and != ignore_index) of the logit C_v . E_i,
 *   computed as C_v . (sum_i E_i) -- the statistic "Cut Your Losses ...",
 *   section "Vocabulary Sorting", accumulates (its average is sums / count).
 *   Deterministic: fp32 column sums in a fixed order, then fp32 dot products
 *   in a fixed order.
 * cce_vocab_order: perm (int32 [V], written) = the stable ascending order of
 *   keys (fp32 [V], device): perm[j] is the token at position j; equal keys
 *   (-0.0 equals +0.0) keep increasing token id.  The order of NaN keys is
 *   unspecified.  A least-significant-digit radix sort, 4 passes of 8 bits.
 * workspace: >= cce_vocab_sort_workspace_bytes(N, D, V) bytes, scratch (for
 *   cce_vocab_order any N >= 1, D >= 8 with D % 8 == 0 gives a large enough
 *   figure).  Same argument checks and status codes as the other calls; E, C
 *   and workspace 16-byte aligned, keys / sums / perm 4-byte aligned.
 */
size_t cce_vocab_sort_workspace_bytes(int64_t N, int64_t D, int64_t V);
cce_status cce_vocab_logit_sums(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                                int64_t ignore_index, float* sums, void* workspace, size_t ws_bytes, void* stream);
cce_status cce_vocab_order(const float* keys, int64_t V, int32_t* perm, void* workspace, size_t ws_bytes,
                           void* stream);

/*
 * Single call: the loss and both gradients in one pass ("fused-linear-cross-
 * entropy" page, section "2. Fused Linear Cross-Entropy (FLCE)": per token
 * chunk, the logits, then loss and dlogits = softmax - onehot, then
 * dx = dlogits C and dw += dlogits^T x; the autograd backward only scales).
 * dE and dC are the gradients of the reduced loss for a unit upstream
 * gradient; multiply them by the real one with cce_scale_grads (both are
 * linear in it).  Only CCE_RED_SUM and CCE_RED_MEAN (a scalar upstream
 * gradient); CCE_RED_NONE returns CCE_ERR_ARG.
 *
 * The rows that take part (target in [0, V) and not ignore_index) are
 * compacted on the device first ("Cut Your Losses ...", Table A1: removing
 * ignored tokens), and only they go through the GEMMs.  They are processed in
 * chunks of Nc rows (a multiple of 256) whose logits, staged as fp16
 * [Nc][V rounded up to 256] (each logit minus its row's max over a 32-column
 * chunk), fit in max_staging_bytes (0: 2 GiB; at least one 256-row chunk).
 * Nothing is recomputed: the chunk's logits are computed once (6 n D V flops
 * for n rows taking part, against 8 N D V for cce_forward + cce_backward), at
 * the cost of the staging traffic.  The filter (filter_eps, filter_flags as
 * in cce_backward_ex; CCE_SORT_VOCAB is not accepted) works on tiles of 128
 * consecutive compact rows x 128 vocabulary entries, as in cce_backward.
 * With more than one chunk dC is accumulated in an fp32 buffer in the
 * workspace (the last chunk adds it and writes bf16); dE always goes through
 * fp32 slabs.
 *
 *   loss   [1] fp32 (written).
 *   lse    [N] fp32 (written) or NULL: the LSE of rows that take part, 0 on
 *          the others.
 *   dE     [N, D] bf16, dC [V, D] bf16 (written; ignored rows of dE are +0).
 *   workspace >= cce_loss_and_grad_workspace_bytes(N, D, V, max_staging_bytes).
 *   dev_stats  optional device int64[2]: {tiles, skipped tiles} over all chunks.
 * Checks and status codes as for the other calls.  Deterministic.
 */
size_t cce_loss_and_grad_workspace_bytes(int64_t N, int64_t D, int64_t V, size_t max_staging_bytes);
cce_status cce_loss_and_grad(const void* E, const void* C, const int64_t* x, int64_t N, int64_t D, int64_t V,
                             int64_t ignore_index, int reduction, float softcap, float filter_eps, int filter_flags,
                             size_t max_staging_bytes, float* loss, float* lse, void* dE, void* dC, void* workspace,
                             size_t ws_bytes, int32_t* dev_err, int64_t* dev_stats, void* stream);

/* dE *= g and dC *= g for bf16 arrays of nE and nC elements (multiples of 8,
 * 16-byte aligned), g = *grad_out (device fp32); nothing is written when
 * g == 1.  The backward of the single call. */
cce_status cce_scale_grads(void* dE, int64_t nE, void* dC, int64_t nC, const float* grad_out, void* stream);

/* Memory accounting (host arithmetic, no GPU).  Reproduces the page's memory
 * table ("Cut Cross-Entropy: Training Loss Without the Logit Matrix ...",
 * section "The memory numbers hold up"): the fp32 N x V logit buffer that the
 * method avoids, the bf16 gradients dC and dE, and this library's workspaces
 * ("extra" device memory beyond inputs and outputs). */
typedef struct {
  uint64_t logits_fp32_bytes;   /* N * V * 4: never allocated by this library */
  uint64_t dE_bytes;            /* N * D * 2 */
  uint64_t dC_bytes;            /* V * D * 2 */
  uint64_t lse_bytes;           /* N * 4 */
  uint64_t fwd_workspace_bytes; /* cce_forward_workspace_bytes() */
  uint64_t bwd_workspace_bytes; /* cce_backward_workspace_bytes() */
  uint64_t bwd_chunk_cols;      /* vocabulary columns per backward chunk */
  uint64_t fwd_vocab_splits;    /* vocabulary splits of the forward partials */
} cce_memory_report;

cce_status cce_memory_accounting(int64_t N, int64_t D, int64_t V, cce_memory_report* out /* host */);

/* Self-test of the failure path of every in-kernel wait.  Launches one
 * thread that waits, through the same bounded wait the GEMM pipelines use, on
 * an mbarrier nothing arrives on; after timeout_us (1 .. 10^7) microseconds the
 * wait gives up and ORs CCE_DEVERR_TIMEOUT into *dev_err (device memory).  No
 * fault, no hang: the context stays usable.  Asynchronous on `stream`. */
cce_status cce_selftest_wait_timeout(int32_t* dev_err, uint32_t timeout_us, void* stream);

/* Self-test of the abort path between the two CTAs of a CTA pair (the
 * forward, recompute and gradient GEMMs run as clusters of two CTAs whose
 * waits depend on each other).  Launches one cluster of two CTAs running the pair's
 * handshake: the odd CTA arrives on a barrier of the even CTA, which answers
 * on a barrier of the odd CTA.  With hold = 1 the odd CTA holds its arrive
 * back: the even CTA's bounded wait runs out after timeout_us (1 .. 10^7)
 * microseconds, the odd CTA's wait for the answer runs out as well, the odd
 * CTA waits the GEMM's bounded 10 ms grace for copies in flight, and both
 * CTAs meet at the final cluster barrier and exit; CCE_DEVERR_TIMEOUT is
 * OR-ed into *dev_err.  With hold = 0 the handshake completes and *dev_err is
 * left alone.  No fault, no hang: the context stays usable.  Other hold
 * values return CCE_ERR_ARG.  Asynchronous on `stream`. */
cce_status cce_selftest_pair_timeout(int32_t* dev_err, uint32_t timeout_us, int hold, void* stream);

/* Test hook of the gradient GEMM as CTA pairs.  A work item carries the
 * survival map of its K range as 64-bit words (one bit per 128 x 128 filter
 * tile), at most 40; a longer K range (more than 327,680 rows taking part in
 * a dC tile) is walked on the maps by the TMA producer instead.  This sets
 * the most words an item may carry to `words` (1 .. 40; any other value
 * restores 40) for the calls that start after it, so tests reach the long
 * path at small sizes, and returns the previous setting.  Process-wide; not
 * meant for production use.  No device work. */
int cce_selftest_pair_map_words(int words);

/* Test hook of the gradient GEMM's layout.  With D tiles 256 wide the
 * gradient GEMM can run as CTA pairs (M = 256 over two row blocks, which
 * run the union of their surviving K-blocks) or one CTA per tile; with the
 * filter on both are launched and the chunk's count of kept filter tiles
 * picks one on the device (pairs from 80% kept).  layout = 1 always runs the
 * pairs where they apply, 2 always one CTA per tile, 0 (or any other value)
 * restores the choice, for the calls that start after it; returns the
 * previous setting.  Process-wide; not meant for production use.  No device
 * work. */
int cce_selftest_grad_layout(int layout);

/* Human-readable name of a status. */
const char* cce_status_string(cce_status s);

/* ABI version (major * 100 + minor): 101.  Minor 1 added cce_backward_ex2,
 * cce_backward_workspace_bytes_ex2, cce_backward_chunk_cols and the
 * selftest entry points cce_selftest_pair_timeout, cce_selftest_pair_map_words
 * and cce_selftest_grad_layout; nothing of 1.0 changed. */
int cce_abi_version(void);

/* Number of kernels this library has launched in this process. */
uint64_t cce_kernel_launch_count(void);

/* Phase timing for measurement.  When enabled, every cce_forward /
 * cce_backward records CUDA events on its stream around each kernel phase.
 * cce_profile_read synchronises on those events and returns, per phase, the
 * summed milliseconds and the number of launches since the last reset.
 * Phases: 0 fwd_lse_gemm, 1 fwd_combine, 2 bwd_prep, 3 bwd_recompute_g,
 * 4 bwd_grad_gemm (dC and dE of a vocabulary chunk, one launch), 5 bwd_finalize,
 * 6 bwd_vocab_sort (with CCE_SORT_VOCAB: sums, order, target remap, and the
 * per-chunk gather of C), 7 single_g_pass (cce_loss_and_grad: staged logits to
 * G; its logit GEMMs count as phase 0, combines as 1, row count as 2,
 * gradient GEMMs as 4, finalisation as 5). */
#define CCE_NUM_PHASES 8
cce_status cce_profile_enable(int enable);
cce_status cce_profile_reset(void);
cce_status cce_profile_read(double* ms /* host [CCE_NUM_PHASES] */, int64_t* launches /* host [CCE_NUM_PHASES] */);
const char* cce_profile_phase_name(int phase);

#ifdef __cplusplus
}
#endif

#endif /* CCE_GB300_H */
