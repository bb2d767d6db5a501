/*
 * kvsel — window-attention prompt-token scoring and top-k KV selection on one GPU.
 *
 * C ABI of libkvsel.so.  Every pointer argument is caller-owned; device
 * pointers are marked [device], host pointers [host].  No call allocates or
 * frees device memory and no call synchronises a stream except
 * kvsel_read_device_error() and kvsel_trace_read().  Calls are asynchronous
 * on the stream passed in; the library keeps no per-call state, so calls with
 * distinct workspaces may run concurrently from several host threads.
 *
 * Stream capture.  The calls of a step (scoring, aggregation, selection,
 * compaction, page table, attention) enqueue only kernels and memsets on the
 * stream and read host arguments at call time, so a step can be captured into
 * a CUDA graph (in any capture mode) and replayed; a replay reads the device
 * buffers as they are then, with the host arguments of the captured call.
 * kvsel_read_device_error() and kvsel_trace_read() synchronise and are not
 * for capture.
 *
 * Arguments are checked on the host before any launch; a rejected call
 * returns a status and launches nothing.  A launch failure returns
 * KVSEL_ERR_CUDA.  Errors that only the device can see (a bounded wait that
 * ran out, an index out of range, a device-resident length out of range) are
 * recorded in an error word at the start of the workspace and read back with
 * kvsel_read_device_error().
 *
 * Prefix lengths on the device.  A caller whose ragged lengths live in device
 * memory (CompactAttention, 'Future directions': page-table metadata built on
 * the kernel side, with no CPU-GPU synchronisation) sets
 * kvsel_desc.prefix_lens_dev and prefix_len_max instead of prefix_lens.  Each
 * call then builds its per-sequence offsets on the device (one small kernel
 * per call, on the call's stream) and sizes its grids for prefix_len_max.
 * What changes for the caller:
 *   - the layouts stay packed by the real lengths, but every buffer must have
 *     room for every sequence at prefix_len_max (the kernels' tensor maps and
 *     grids are sized for the bound);
 *   - every call needs a workspace, including kvsel_compact,
 *     kvsel_compact_layers and kvsel_prefill_attention;
 *   - checks that depend on a length (1 <= L_b <= prefix_len_max; kvsel_topk's
 *     k <= L_b and its page rules; kvsel_pagetable's n_kvblk, then read from
 *     device memory) run on the device: a failed check records
 *     KVSEL_ERR_INVALID_ARG (detail: the sequence) in the error word and that
 *     call's kernels leave their outputs unwritten.
 *
 * Layouts (bf16 = IEEE bfloat16 bit pattern in uint16 storage, row-major,
 * sequences of a batch packed one after another in batch order):
 *   q            [batch][n_layers][h_q][W][d]                     bf16
 *   k, v         per sequence b: [n_layers][h_kv][L_b + W][d]     bf16
 *   scores       per sequence b: [n_layers][h_kv][L_b]            fp32
 *   page_scores  per sequence b: [n_layers][h_kv][ceil(L_b / P)]  fp32
 * Key row t of sequence b is absolute prompt position t: rows 0..L_b-1 are
 * the prefix, rows L_b..L_b+W-1 the observation window whose queries are q.
 * Query head h reads KV head g = h / (h_q / h_kv).
 */
#ifndef KVSEL_H
#define KVSEL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KVSEL_API __attribute__((visibility("default")))
#else
#define KVSEL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVSEL_OK = 0,
  KVSEL_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shape */
  KVSEL_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  KVSEL_ERR_WORKSPACE = 3,     /* workspace null, misaligned or smaller than kvsel_workspace_size() */
  KVSEL_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  KVSEL_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
  KVSEL_ERR_DEVICE = 6         /* the device found an index out of range */
} kvsel_status;

/* group_reduce / page_reduce: sum, max, or (group_reduce only) the mean over the G * W rows of a group */
enum { KVSEL_REDUCE_SUM = 0, KVSEL_REDUCE_MAX = 1, KVSEL_REDUCE_MEAN = 2 };
/* pool_type: max-pooling or average pooling (the mean over the in-range neighbours) */
enum { KVSEL_POOL_MAX = 0, KVSEL_POOL_AVG = 1 };
/* score_mode: post-softmax window probabilities, or the pre-softmax scaled logits */
enum { KVSEL_SCORE_SOFTMAX = 0, KVSEL_SCORE_LOGITS = 1 };
/* kvsel_aggregate: what happens across layers and across KV heads */
enum { KVSEL_LAYERS_EACH = 0, KVSEL_LAYERS_L1_MEAN = 1, KVSEL_LAYERS_MAX = 2 };
enum { KVSEL_HEADS_EACH = 0, KVSEL_HEADS_SUM = 1 };

#define KVSEL_MAX_BATCH 128
#define KVSEL_MAX_WINDOW 64
#define KVSEL_MAX_ROWS 256          /* (h_q / h_kv) * window */
#define KVSEL_MAX_PAGE 256
#define KVSEL_WS_ALIGN 256          /* required workspace alignment in bytes */

/* Shape and reduction modes shared by every call. */
typedef struct {
  int32_t n_layers;            /* >= 1 */
  int32_t h_q;                 /* query heads, multiple of h_kv */
  int32_t h_kv;                /* KV heads >= 1 */
  int32_t head_dim;            /* d: 64 or 128 */
  int32_t window;              /* W: 1 .. KVSEL_MAX_WINDOW; (h_q / h_kv) * W <= KVSEL_MAX_ROWS */
  int32_t batch;               /* sequences: 1 .. KVSEL_MAX_BATCH */
  const int64_t* prefix_lens;  /* [host] [batch] prefix lengths L_b >= 1, L_b + W < 2^31; or NULL with
                                  prefix_lens_dev */
  int32_t group_reduce;        /* KVSEL_REDUCE_SUM, _MAX or _MEAN over the query heads of a group */
  int32_t pool_k;              /* odd pool width, 1 (none) .. 63 */
  int32_t page_size;           /* P: 1 = token mode, 2 .. KVSEL_MAX_PAGE = page mode */
  int32_t page_reduce;         /* KVSEL_REDUCE_MAX or KVSEL_REDUCE_SUM over the tokens of a page */
  int32_t pool_type;           /* KVSEL_POOL_MAX (0) or KVSEL_POOL_AVG */
  int32_t score_mode;          /* KVSEL_SCORE_SOFTMAX (0) or KVSEL_SCORE_LOGITS */
  const int64_t* prefix_lens_dev;  /* [device] [batch] prefix lengths, or NULL (prefix_lens is used);
                                      exactly one of prefix_lens / prefix_lens_dev is set */
  int64_t prefix_len_max;      /* with prefix_lens_dev: bound of every L_b (>= 1, + W < 2^31); sizes the
                                  workspace, the grids and the buffers the caller provides */
} kvsel_desc;

/* Bytes of device workspace the calls below need for this descriptor (any of them). */
KVSEL_API kvsel_status kvsel_workspace_size(const kvsel_desc* desc, size_t* bytes);

/*
 * kvsel_score — window-query attention scores of every prefix token.
 *
 * ClusterAttn: KV Cache Compression under Intrinsic Attention Clustering,
 * 'Background and key observations', feature aggregation: the W window
 * queries attend to all prompt keys through a causal mask inside the window
 * (row j sees prefix keys and window keys 0..j), QK^T / sqrt(d), softmax over
 * the full row, then the post-softmax mass is summed over the window rows for
 * each prefix column.  The per-head column mass is reduced over the query
 * heads of each GQA group (sum as in CLAA's FastKV-style window scoring,
 * max as in DELTA's head-aware scoring, or the mean over the group's rows as
 * LookaheadKV averages its lookahead rows), pooled with width pool_k over
 * prefix positions (CLAA, 'Oracle construction': 1-D pooling, kernel 7; max
 * or average, out-of-range neighbours ignored), and, in page mode, reduced to
 * page scores over P consecutive tokens (DELTA, 'Key designs' 2 and 3).
 * With score_mode KVSEL_SCORE_LOGITS the softmax is skipped and the scaled
 * logits are summed instead (CLAA, 'Three representative token-ranking
 * methods': GemFilter's pre-softmax score of the last prompt token, W = 1);
 * that mode makes one pass over K instead of two.
 *
 *   q, k         [device] bf16, layouts above; 16-byte aligned
 *   scores       [device] fp32 out: pooled token scores (raw group scores when pool_k == 1)
 *   page_scores  [device] fp32 out in page mode (may be NULL in token mode)
 *   ws           [device] workspace of ws_bytes >= kvsel_workspace_size(), KVSEL_WS_ALIGN aligned
 */
KVSEL_API kvsel_status kvsel_score(const kvsel_desc* desc, const void* q, const void* k,
                         float* scores, float* page_scores,
                         void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_prefill_attention — causal attention of every prompt row, with what the window scoring needs.
 *
 * o_i = sum over keys t <= i of softmax(q_i k_t / sqrt(d)) v_t for every row i of every query head
 * (GQA map h -> h / (h_q / h_kv)), on the tensor cores.  CLAA, 'Complete flow and cost' (engineering
 * detail 1): the keys that score the observation window are the prefill's own; the prefill's softmax
 * forms each row's log-sum-exp, which is the first of the scoring's two passes for the window rows.
 * So the call also writes the window rows' lse (base 2, units of z log2(e) / sqrt(d), in the order
 * kvsel_score_from_lse reads) and the window queries; kvsel_score_from_lse then scores with one pass.
 *
 *   q, o     [device] bf16, per sequence b: [n_layers][h_q][L_b + W][d]; d = 128
 *   k, v     [device] bf16 caches, layout above
 *   lse      [device] fp32 out, natural-log lse of every row, layout of q without d (nullable)
 *   lse_win  [device] fp32 out [batch][n_layers][h_kv][(h_q / h_kv) * W], row (h_local, j)
 *   q_win    [device] bf16 out [batch][n_layers][h_q][W][d] (the layout kvsel_score reads)
 *   ws       [device] workspace or NULL (error word for bounded waits)
 */
KVSEL_API kvsel_status kvsel_prefill_attention(const kvsel_desc* desc, const void* q, const void* k, const void* v,
                                               void* o, float* lse, float* lse_win, void* q_win, void* ws,
                                               cudaStream_t stream);

/*
 * kvsel_score_from_lse — kvsel_score with the window rows' lse given (from kvsel_prefill_attention).
 *
 * Computes what kvsel_score computes (softmax mode) with the second pass only: the column mass of
 * the window probabilities 2^(z log2(e) / sqrt(d) - lse) for every prefix key, the group reduce,
 * pooling and page reduce.  One read of the prefix keys instead of two.
 *
 *   q_win    [device] bf16 window queries, layout above
 *   lse_win  [device] fp32, as kvsel_prefill_attention writes it
 *   other arguments as for kvsel_score
 */
KVSEL_API kvsel_status kvsel_score_from_lse(const kvsel_desc* desc, const void* q_win, const void* k,
                                            const float* lse_win, float* scores, float* page_scores, void* ws,
                                            size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_combine_layers — cross-layer aggregation of raw group scores.
 *
 * Each layer's scores of a (sequence, KV head) row are L1-normalised over the
 * prefix (LookaheadKV, 'KL divergence and ListNet': s / ||s||_1), the mean is
 * taken over layers layer_lo..layer_hi inclusive (CLAA, decision 3: one score
 * per token aggregated over several layers), and the result is pooled with
 * desc->pool_k / desc->pool_type.  Same as kvsel_aggregate with
 * KVSEL_LAYERS_L1_MEAN and KVSEL_HEADS_EACH.
 *
 *   scores    [device] fp32 raw group scores (kvsel_score with pool_k = 1), layout above
 *   combined  [device] fp32 out, per sequence b: [h_kv][L_b]
 *   ws        [device] workspace (holds the per-layer L1 norms)
 */
KVSEL_API kvsel_status kvsel_combine_layers(const kvsel_desc* desc, const float* scores,
                                  int32_t layer_lo, int32_t layer_hi, float* combined,
                                  void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_aggregate — reduce raw group scores across KV heads and layers, then pool.
 *
 * For each sequence, over layers layer_lo..layer_hi (inclusive) of raw group
 * scores (kvsel_score with pool_k = 1):
 *   head_op  KVSEL_HEADS_EACH keeps every KV head; KVSEL_HEADS_SUM sums all KV
 *            heads of a layer (the sum over all attention heads that FastKV,
 *            CLAA and GemFilter rank with; CLAA, decision 2);
 *   layer_op KVSEL_LAYERS_EACH keeps every layer of the range;
 *            KVSEL_LAYERS_L1_MEAN L1-normalises each layer's row over the prefix
 *            (LookaheadKV, 'KL divergence and ListNet') and averages the range;
 *            KVSEL_LAYERS_MAX takes the token-wise max over the range (CLAA,
 *            decision 3, Eq. 6, at the pruning layer);
 * then pools with desc->pool_k / desc->pool_type.  Token scores only.
 *
 *   scores  [device] fp32 raw group scores, per sequence b: [n_layers][h_kv][L_b]
 *   out     [device] fp32, per sequence b: [n_l][n_h][L_b], n_l = layer_hi - layer_lo + 1
 *           (EACH) or 1, n_h = h_kv (EACH) or 1; sequences packed in batch order
 *   ws      [device] workspace (holds the L1 norms)
 */
KVSEL_API kvsel_status kvsel_aggregate(const kvsel_desc* desc, const float* scores, int32_t layer_lo,
                                       int32_t layer_hi, int32_t layer_op, int32_t head_op, float* out,
                                       void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_select — top-k selection over any rows of scores, ties to the lower index.
 *
 * As kvsel_topk (below), over `rows` score rows per sequence: per sequence b,
 * scores [rows][n] with n = L_b (token mode) or ceil(L_b / P) (page mode),
 * sequences packed in batch order.  With append_window == 0 the window
 * positions (or window pages) are not appended — for windows whose keys are
 * not part of the prompt to keep, such as LookaheadKV's lookahead rows,
 * which take no part in decoding ('Method steps').
 *
 *   idx_out  [device] int32 out [batch][rows][n_sel], n_sel = k (+ W with the
 *            window, token mode) or k + n_recent (+ W / P with the window, page mode)
 */
KVSEL_API kvsel_status kvsel_select(const kvsel_desc* desc, const float* scores, int32_t rows, int32_t k,
                                    int32_t n_recent, int32_t append_window, int32_t* idx_out,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_topk — top-k selection per (sequence, layer, KV head) row, ties to the lower index.
 *
 * Token mode (desc->page_size == 1): the k prefix tokens of highest score,
 * in ascending position, then the window positions L_b .. L_b+W-1 (ClusterAttn,
 * 'Method details': the compressed prefix is joined with the window).
 * Page mode: the last n_recent prefix pages are kept and the k highest-scoring
 * of the other prefix pages are added (DELTA, 'Key designs' 2: recency pages
 * union top pages of the rest), in ascending order, then the W / P pages of
 * the window.  Page mode requires W % P == 0, and n_recent >= 1 when
 * L_b % P != 0 (so the page shared by prefix and window is kept once).
 *
 *   scores   [device] fp32 per sequence b: [layers][h_kv][n] with n = L_b (token mode)
 *            or ceil(L_b / P) (page mode); layers = desc->n_layers, or 1 for the
 *            output of kvsel_combine_layers
 *   idx_out  [device] int32 out [batch][layers][h_kv][n_sel], n_sel = k + W (token)
 *            or k + n_recent + W / P (page): token positions or page numbers
 */
KVSEL_API kvsel_status kvsel_topk(const kvsel_desc* desc, const float* scores, int32_t layers,
                        int32_t k, int32_t n_recent, int32_t* idx_out,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_compact — gather the kept K and V rows into a compacted cache.
 *
 * CLAA, 'Complete flow and cost': each layer's cache keeps only the K and V
 * rows of the selected tokens; ClusterAttn, 'Method details', keeps the window
 * rows with them.  Token mode copies row idx[r]; page mode copies the P rows
 * of page idx[r] (rows past L_b + W are written as zero).  A bit copy:
 * outputs equal inputs exactly.
 *
 *   k, v          [device] bf16 caches, layout above; either may instead be pinned
 *                 host memory mapped at the same address (cudaHostAlloc, or
 *                 cudaHostRegister with cudaHostRegisterMapped): the kernel then
 *                 reads only the kept rows over the host link, so a cache held on
 *                 the host never has to be copied whole.  Any other pointer (pageable
 *                 host memory, another device's memory) is rejected with
 *                 KVSEL_ERR_INVALID_ARG before the launch.
 *   idx           [device] int32 [batch][idx_layers][h_kv][n_sel] as written by kvsel_topk;
 *                 idx_layers == 1 applies one selection to every layer
 *   k_out, v_out  [device] bf16 out [batch][n_layers][h_kv][n_sel * P][d]
 *   ws            [device] workspace or NULL; an index out of range is not
 *                 followed, its row is zeroed and, with ws, KVSEL_ERR_DEVICE is
 *                 recorded in the error word
 */
KVSEL_API kvsel_status kvsel_compact(const kvsel_desc* desc, const void* k, const void* v,
                           const int32_t* idx, int32_t idx_layers, int32_t n_sel,
                           void* k_out, void* v_out, void* ws, cudaStream_t stream);

/*
 * kvsel_compact_layers — kvsel_compact over a range of layers, with selections shared by heads.
 *
 * Compacts layers layer_lo .. layer_lo + n_layers_out - 1 of the caches (CLAA,
 * 'Three design decisions', decision 1: the first m layers keep their full
 * cache and are not compacted).  idx is [batch][idx_layers][idx_heads][n_sel]:
 * idx_layers == 1 applies one selection to every compacted layer, otherwise
 * idx_layers == n_layers_out and row i serves layer layer_lo + i; idx_heads == 1
 * applies one selection to every KV head (the all-head scores of CLAA,
 * FastKV and GemFilter rank tokens once per layer), otherwise idx_heads == h_kv.
 *
 *   k, v          as for kvsel_compact (device, or mapped pinned host memory)
 *   k_out, v_out  [device] bf16 out [batch][n_layers_out][h_kv][n_sel * P][d]
 *   ws            [device] workspace or NULL (errors as for kvsel_compact)
 */
KVSEL_API kvsel_status kvsel_compact_layers(const kvsel_desc* desc, const void* k, const void* v,
                                            const int32_t* idx, int32_t idx_layers, int32_t idx_heads,
                                            int32_t layer_lo, int32_t n_layers_out, int32_t n_sel,
                                            void* k_out, void* v_out, void* ws, cudaStream_t stream);

/*
 * kvsel_attend — attention of a few query rows per head over the KV rows a table selects, in place.
 *
 * CompactAttention, 'Method steps' (3): the per-group block list T[b,g] (kv_indptr / kv_indices,
 * as kvsel_pagetable writes it) goes to a paged dense-attention kernel that reads the selected
 * blocks of the KV-head-major cache where they are, with no copy; DELTA, 'Overall framework':
 * sparse layers attend only over the selected page set (the dense page table of kvsel_topk in page
 * mode).  For each table row (b, layer, g) and each of the n_q query rows of each of the G query
 * heads of group g: o = softmax(q K_sel^T / sqrt(d)) V_sel over every row of every listed block
 * (block j covers rows j*block .. j*block + block - 1; rows past L_b + W do not exist), with no
 * causal mask (decode-style queries come after every selected key).  A row that selects nothing
 * gives o = 0.
 *
 *   q           [device] bf16 [batch][n_layers][h_q][n_q][d]; (h_q / h_kv) * n_q <= 32
 *   k, v        [device] bf16 caches, layout above
 *   kv_indptr   [device] int32 [batch * n_layers * h_kv + 1] (CSR), or NULL: row r's list is
 *               kv_indices[r * n_per_row .. (r + 1) * n_per_row) (a dense table)
 *   kv_indices  [device] int32 block ids, or NULL together with kv_indptr: every block of the
 *               row's cache in order (dense attention over the whole cache)
 *   block       rows per block, 1 .. KVSEL_MAX_PAGE
 *   max_blocks  upper bound of any row's list length (sizes the split of each row's work)
 *   o           [device] fp32 out [batch][n_layers][h_q][n_q][d]
 *   ws          [device] workspace of kvsel_attend_workspace_size() bytes (partials of the splits);
 *               a block id whose first row does not exist is skipped and KVSEL_ERR_DEVICE recorded.
 *               The split count, and with it the size, depends on how many warps the current device
 *               keeps resident: query the size on the device the call runs on.
 *
 * Arithmetic: for up to 8 query rows per table row the logits are bf16 products accumulated in fp32
 * (tensor cores) and P V takes P to ~16 significant bits (a bf16 high and low part); more rows use
 * fp32 FMA throughout.
 */
KVSEL_API kvsel_status kvsel_attend_workspace_size(const kvsel_desc* desc, int32_t n_q, int32_t block,
                                                   int32_t max_blocks, size_t* bytes);
KVSEL_API kvsel_status kvsel_attend(const kvsel_desc* desc, const void* q, int32_t n_q, const void* k,
                                    const void* v, const int32_t* kv_indptr, const int32_t* kv_indices,
                                    int32_t n_per_row, int32_t block, int32_t max_blocks, float* o, void* ws,
                                    size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_claa_shape / kvsel_claa_select — the CLAA schedule over one prompt.
 *
 * CLAA, 'Three design decisions': decision 1, the first m layers (defer) keep their full cache;
 * decision 2, every later layer up to the pruning layer l_p scores the prompt with its observation
 * window (post-softmax probabilities summed over the window rows and all heads); decision 3 (Eq. 6),
 * the per-layer scores of the last n layers (the rolling buffer, layers max(m, l_p - n + 1) .. l_p)
 * are aggregated token-wise by their maximum.  'Complete flow and cost': each scored layer keeps
 * topk(score, keep_rate) of the prefix (k = floor(r L + 1/2), clipped to [0, L]) plus the window and
 * gathers its cache to those rows; at l_p the pooled aggregate picks the sequence prune index.
 * Pooling is desc->pool_k / pool_type ('Experimental setup': average pooling, kernel 7).
 *
 * The descriptor covers every layer of the prompt (batch 1, host prefix length, token mode,
 * group_reduce KVSEL_REDUCE_SUM, score_mode KVSEL_SCORE_SOFTMAX).  kvsel_claa_shape returns the
 * sizes the outputs need; kvsel_claa_select runs the schedule:
 *   q, k, v        [device] bf16, layouts above, all n_layers layers; v is only gathered, so it
 *                  may be mapped pinned host memory (as for kvsel_compact)
 *   scores         [device] fp32 out [n_scored][h_kv][L]: raw group scores of layers m .. l_p
 *   layer_scores   [device] fp32 out [n_scored][L]: pooled all-head score of each scored layer
 *   prune_scores   [device] fp32 out [L]: pooled token-wise max over the buffer
 *   idx            [device] int32 out [n_scored][n_sel]: each scored layer's kept rows
 *   prune_idx      [device] int32 out [n_sel]: the prune index
 *   k_out, v_out   [device] bf16 out [n_scored][h_kv][n_sel][d]: compacted caches of layers m .. l_p
 *   ws             [device] workspace of at least shape.ws_bytes
 */
typedef struct {
  int32_t defer;          /* m: layers 0 .. m - 1 are neither scored nor compacted */
  int32_t prune_layer;    /* l_p: m <= l_p < n_layers */
  int32_t n_buffer;       /* n >= 1: layers in the rolling buffer */
  double keep_rate;       /* r in [0, 1]: fraction of the prefix kept */
} kvsel_claa_params;

typedef struct {
  int32_t n_scored;       /* l_p - m + 1 */
  int32_t buffer_lo;      /* first buffered layer, max(m, l_p - n + 1); the last is l_p */
  int32_t k;              /* prefix tokens kept per selection */
  int32_t n_sel;          /* entries per selection: k + W */
  size_t ws_bytes;        /* workspace kvsel_claa_select needs */
} kvsel_claa_shape_t;

KVSEL_API kvsel_status kvsel_claa_shape(const kvsel_desc* desc, const kvsel_claa_params* p, kvsel_claa_shape_t* out);
KVSEL_API kvsel_status kvsel_claa_select(const kvsel_desc* desc, const kvsel_claa_params* p, const void* q,
                                         const void* k, const void* v, float* scores, float* layer_scores,
                                         float* prune_scores, int32_t* idx, int32_t* prune_idx, void* k_out,
                                         void* v_out, void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_pagetable — per-group KV block table from a 2-D block mask.
 *
 * CompactAttention: Accelerating Chunked Prefill with Block-Union KV
 * Selection, 'Method steps' (2): Q-block union Mbar[b,h,j] = OR_i M[b,h,i,j],
 * intra-group union G[b,g,j] = OR over the heads h of group g, and
 * T[b,g] = { j : G[b,g,j] = 1 } in ascending order, written as CSR
 * (kv_indptr / kv_indices) over rows (b, layer, g).
 *
 *   mask        [device] uint8 [batch][n_layers][h_q][n_qblk][n_kvblk_max], nonzero = selected
 *   n_kvblk     [host] [batch] KV blocks of each sequence (<= n_kvblk_max); mask
 *               entries at j >= n_kvblk[b] are ignored.  [device] when the descriptor's
 *               prefix lengths are on the device (prefix_lens_dev)
 *   kv_indptr   [device] int32 out [batch * n_layers * h_kv + 1]
 *   kv_indices  [device] int32 out, capacity batch * n_layers * h_kv * n_kvblk_max
 */
KVSEL_API kvsel_status kvsel_pagetable(const kvsel_desc* desc, const uint8_t* mask, int32_t n_qblk,
                             int32_t n_kvblk_max, const int32_t* n_kvblk,
                             int32_t* kv_indptr, int32_t* kv_indices,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * kvsel_score_noalloc — kvsel_score for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers with no
 * way to obtain a workspace: a plugin inside a host program that owns all of
 * the GPU's memory, or a latency-critical caller that must not pay
 * cudaMalloc's device-wide synchronisation.  It computes exactly what
 * kvsel_score computes, with the scratch of the two scoring passes in an
 * array inside the library of KVSEL_NOALLOC_SCRATCH_BYTES, which every GPU
 * that loads the library holds until the process exits.  It allocates and
 * frees nothing.
 *
 * The first call made while a device is current looks up that array's device
 * address (cudaGetSymbolAddress) and caches it for the life of the process;
 * make that first call before any stream capture.  cudaDeviceReset after it
 * is not supported (the module may then load at another address and the
 * cached one would be stale).  The stream must belong to the current device.
 * All calls share the one array: calls whose work overlaps on the GPU (two
 * streams, or two host threads) race and give undefined results.  Arguments
 * are checked as kvsel_score checks them, and a descriptor whose
 * kvsel_workspace_size() exceeds KVSEL_NOALLOC_SCRATCH_BYTES is rejected with
 * KVSEL_ERR_WORKSPACE; a rejected call launches nothing and enqueues nothing.
 *
 * Errors only the device sees (a bounded wait that ran out) go to the error
 * word at the start of the array, which each call clears first; read it with
 * kvsel_noalloc_read_device_error() on the call's stream before the next call.
 */
#define KVSEL_NOALLOC_SCRATCH_BYTES (32u << 20)
KVSEL_API kvsel_status kvsel_score_noalloc(const kvsel_desc* desc, const void* q, const void* k,
                                           float* scores, float* page_scores, cudaStream_t stream);

/* Reads (stream-synchronising) and clears the error word of the current device's built-in scratch:
 * the status of the last kvsel_score_noalloc call on that device, or KVSEL_OK. */
KVSEL_API kvsel_status kvsel_noalloc_read_device_error(cudaStream_t stream);

/*
 * kvsel_selftest_bounded_wait — exercises the bounded device wait used by every pipelined kernel.
 *
 * The pages have no counterpart to this call; it exists so that failure reporting can be tested
 * without a real fault.  It launches one CTA that waits on a shared-memory mbarrier with the same
 * wait routine the scoring kernels use.  With arrive == 0 nothing completes the barrier, the wait
 * gives up after `polls` polls (1 .. 2^22) and KVSEL_ERR_TIMEOUT is recorded in the error word of
 * `ws` (read it with kvsel_read_device_error); with arrive != 0 a second thread completes the
 * barrier and nothing is recorded.
 */
KVSEL_API kvsel_status kvsel_selftest_bounded_wait(void* ws, uint32_t polls, int32_t arrive, cudaStream_t stream);

/* Reads (stream-synchronising) and clears the device error word of a workspace. */
KVSEL_API kvsel_status kvsel_read_device_error(void* ws, cudaStream_t stream);

KVSEL_API const char* kvsel_status_string(kvsel_status status);
KVSEL_API const char* kvsel_version(void);

/*
 * Tracing.  With tracing on, every kernel launch of the library is bracketed
 * by CUDA events on its stream; kvsel_trace_read() synchronises those events
 * and returns, per kernel name, the launches and the summed milliseconds since
 * the last read.  kvsel_launch_count() counts every kernel launch since load.
 */
typedef struct {
  char name[48];
  int64_t launches;
  double ms;
} kvsel_trace_entry;

KVSEL_API void kvsel_trace_enable(int32_t on);
KVSEL_API kvsel_status kvsel_trace_read(kvsel_trace_entry* out, int32_t capacity, int32_t* n_out);
KVSEL_API int64_t kvsel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KVSEL_H */
