/*
 * hsa.h -- C ABI of libhsa: one decode step of hierarchically pruned, block-sparse
 * attention over a paged KV cache with int8 per-channel-quantised keys, on one GB300
 * GPU (sm_103a).
 *
 * The step (sources, by page title and section):
 *   1. append the new token's key and value to its page and give the key its int8
 *      codes with the stored channel scales;
 *   2. fold the key scales into the query and quantise it (one scale per group of
 *      query heads), score every candidate token exactly in int32 against the int8
 *      keys -- "HCAttention: Extreme KV cache compression via heterogeneous attention
 *      computing for LLMs", abstract and contribution list (quantised keys kept on the
 *      GPU for a global approximate scoring; values fetched late);
 *   3. module 1: cut the context into chunks, score each by its best token, keep the
 *      top-K1; module 2: cut the survivors into 16-token blocks, keep the top-K2 --
 *      InfiniteHiP article (163.com, "韩国通过卸载键值缓存节约英伟达GPU内存，实现18.95倍
 *      解码加速"), section "实现 7.24 倍的端到端解码加速" (modular hierarchical pruning);
 *   4. exact softmax attention over the attention sinks, the recent window and the
 *      kept blocks, from the bf16 K/V, split over many CTAs and merged by log-sum-exp
 *      -- "KV Cache 与长上下文推理", sections "KV Cache 回顾" (decode attention
 *      equation) and "Token Eviction 与 Sparse Attention" (StreamingLLM sinks +
 *      sliding window).
 *
 * Conventions shared by every call:
 *  - Every pointer is a DEVICE pointer unless a flag below says otherwise. The caller
 *    owns every buffer and the stream; the library never allocates or frees memory
 *    (hsa_decode_step's recorded graphs aside: see there), never synchronises (except
 *    hsa_read_device_error, which says so), and never aborts or traps. `stream` is a
 *    cudaStream_t (NULL = legacy default stream).
 *  - Paged cache layout: [num_pages][hkv][page_size=16][head_dim=128], bf16 for K and
 *    V, int8 for the key codes; token t of sequence b lives in page
 *    page_table[b * max_pages_per_seq + t / 16], slot t % 16. page_table is int32
 *    [batch][max_pages_per_seq]; entries past a sequence's last page are never read.
 *  - seq_lens int32 [batch]: N_b, the context INCLUDING the current token.
 *  - Query q: bf16 [batch][hq][128]; query head j uses kv head j / (hq / hkv).
 *  - Candidate region of sequence b: C_b = [sink, N_b - window) (empty when
 *    N_b <= sink + window). Chunks [c*chunk, (c+1)*chunk) and blocks [16k, 16k+16)
 *    are aligned to token 0; only their tokens inside C_b count, and a chunk or block
 *    with no token in C_b is never selected.
 *  - Attended set T_b = [0, min(sink,N)) u [max(N-window, min(sink,N)), N) u
 *    (kept blocks n C_b).
 *  - Ties in either module: the lower index wins. Index lists are ascending and padded
 *    with -1.
 *  - Key scales (int8 reading): s_c = f32(amax_c / 127) over the whole context of one
 *    (sequence, kv head, channel); code = clamp(rint_half_even(f32(k / s_c)), +-127);
 *    s_c = 0 gives code 0. Query: q'_{j,c} = f32(q_{j,c} s_c); A = max |q'| over the
 *    group; sq = f32(A / 127); qq = clamp(rint_half_even(f32(q' / sq)), +-127).
 *    Token score: max over the group of sum_c qq_{j,c} kq_{t,c} (exact int32).
 *  - Workspace: caller-allocated device memory of at least hsa_workspace_bytes(d, op)
 *    bytes, 256-byte aligned, ZERO-FILLED ONCE before its first use. Calls leave the
 *    counters they use at zero again, so one workspace serves any number of calls,
 *    but two calls that run at the same time must not share a workspace. Word 0 of
 *    every workspace is a device error word (see hsa_read_device_error).
 *  - Return value: HSA_OK or an HSA_ERR_* code; on error nothing was launched unless
 *    the code is HSA_ERR_CUDA.
 */
#ifndef HSA_H_
#define HSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum hsa_status {
  HSA_OK = 0,
  HSA_ERR_INVALID_ARG = 1,          /* null pointer, bad size, misaligned pointer */
  HSA_ERR_UNSUPPORTED = 2,          /* head_dim != 128, page/block != 16, group not 1/2/4/8, ... */
  HSA_ERR_CUDA = 3,                 /* a CUDA runtime call or a launch failed */
  HSA_ERR_TIMEOUT = 4,              /* a bounded device wait ran out (reported by the error word) */
  HSA_ERR_WORKSPACE_TOO_SMALL = 5,
  HSA_ERR_DEVICE_CHECK = 6          /* a device-side bounds check failed (bad page-table entry) */
};

/* Problem descriptor. Only the fields an entry point uses need to be valid for it. */
typedef struct hsa_dims {
  int32_t batch;             /* sequences in the step (>= 1) */
  int32_t hq;                /* query heads */
  int32_t hkv;               /* key/value heads; hq % hkv == 0 and hq / hkv in {1, 2, 4, 8} */
  int32_t head_dim;          /* must be 128 */
  int32_t page_size;         /* must be 16 */
  int32_t max_pages_per_seq; /* row length of page_table (>= 1) */
  int32_t num_pages;         /* pages in the pool; every page-table entry read must be < this */
  int32_t chunk;             /* module-1 chunk length in tokens: a positive multiple of 16 */
  int32_t block;             /* module-2 block length in tokens: must be 16 */
  int32_t k1;                /* chunks kept by module 1 (>= 0) */
  int32_t k2;                /* blocks kept by module 2 (>= 0) */
  int32_t sink;              /* leading tokens always attended (>= 0) */
  int32_t window;            /* trailing tokens always attended (>= 0) */
  float sm_scale;            /* softmax scale of q.k; <= 0 selects 1/sqrt(head_dim) */
  int32_t kv_on_host;        /* 1: the bf16 K/V caches given to hsa_attend, dense_decode,
                                hsa_append_kv and hsa_decode_step are PINNED HOST memory
                                (cudaHostAlloc / cudaHostRegister); the kernels read them
                                through the mapped device aliases */
  int32_t chunk0;            /* k0 > 0: length of module 0's coarse chunks, a multiple of chunk */
  int32_t k0;                /* coarse chunks kept by module 0, stacked in front of module 1
                                (which then ranks only the chunks inside them); 0: no module 0 */
  int32_t key_bits;          /* key codes: 0 or 8 = 8-bit (kq int8 [num_pages][hkv][16][128]);
                                4 = 4-bit (scale amax / 7, codes in [-7, 7], two per byte: kq
                                [num_pages][hkv][16][64] bytes, channel 2i in the low nibble) */
  int32_t per_head;          /* 0: the G query heads of a kv head share one selection (token
                                score = max over the group); 1: per-head selection (InfiniteHiP
                                article: every head is pruned on its own): each query head
                                ranks its own scores (same query codes), and every selection
                                array has one row per QUERY head: block_max / tile_max
                                [batch][hq][..], chunk_idx / block_idx [batch][hq][k1 / k2],
                                n_chunks / n_blocks [batch][hq]; the attention of query head
                                j then reads row j. Not with the block cache (UNSUPPORTED). */
  int32_t key_fp8;           /* 0: integer key codes (key_bits); 1: FP8 E4M3 key codes, in the
                                8-bit layout (kq [num_pages][hkv][16][128] bytes; key_bits 0 or
                                8, else UNSUPPORTED): s = f32(amax / 448), code = E4M3 of
                                f32(k / s) rounded to nearest even, saturating at +-448; the
                                query is folded (q' = f32(q * s)) but not quantised and a
                                token's score is the fp32 fused multiply-add chain over the
                                channels in order; block_max / tile_max then hold the scores'
                                order-preserving integer images (bits, negative ones with the
                                magnitude bits flipped) */
  int32_t cache_policy;      /* victims of the GPU block cache (hsa_attend_cached,
                                hsa_decode_step_cached): 0 = least recently used; 1 = least
                                cumulative attention mass (HCAttention: reversible eviction of
                                the least important KV blocks by a cumulative-magnitude
                                criterion); other values INVALID_ARG */
} hsa_dims;

/* Operation ids for hsa_workspace_bytes. */
enum hsa_op {
  HSA_OP_QUANTIZE = 0,
  HSA_OP_SELECT = 1,
  HSA_OP_ATTEND = 2,
  HSA_OP_DENSE = 3,
  HSA_OP_STEP = 4,
  HSA_OP_CACHED = 5
};

/* Workspace bytes `op` needs for descriptor `d` (0 if `d` is invalid). */
size_t hsa_workspace_bytes(const hsa_dims* d, int32_t op);

/* Short English text for a status code (static storage). */
const char* hsa_status_string(int32_t status);

/*
 * Key quantisation (HCAttention abstract: quantised keys kept on the GPU;
 * "KV Cache 与长上下文推理", section "KV Cache 量化": INT8 keys).
 *  mode 0 (FULL): k_scale[b][h][c] = f32(amax / L) over tokens t < N_b, and the codes
 *    of every token t < N_b; slots of a last page past N_b get code 0. Needs
 *    HSA_OP_QUANTIZE workspace. L = 127 for 8-bit codes, 7 for 4-bit (d->key_bits).
 *  mode 1 (APPEND): codes of tokens [append_from, N_b) of every sequence with the
 *    stored k_scale (append_from < 0: each sequence's last token); values beyond the
 *    stored range saturate at +-L. Workspace may be NULL.
 * k_cache: bf16 paged cache (device, or pinned host when d->kv_on_host). kq: paged codes
 * on the device, int8 [num_pages][hkv][16][128], or with d->key_bits == 4 two's-complement
 * nibbles [num_pages][hkv][16][64] bytes (channel 2i in the low nibble of byte i, 2i + 1
 * in the high one). k_scale: f32 [batch][hkv][128].
 */
int32_t hsa_quantize_keys(const hsa_dims* d, const void* k_cache, const int32_t* page_table,
                          const int32_t* seq_lens, int32_t mode, int32_t append_from,
                          int8_t* kq, float* k_scale, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * Decode-step append ("KV Cache 与长上下文推理", section "KV Cache 回顾": each step
 * computes the new token's k and v and appends them to the cache). Writes k_new and
 * v_new (bf16 [batch][hkv][128]) into slot N_b - 1 of each sequence's bf16 caches and
 * the new key's codes into kq (in d->key_bits' format) with the stored k_scale
 * (saturating).
 */
int32_t hsa_append_kv(const hsa_dims* d, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, int8_t* kq, const float* k_scale,
                      const int32_t* page_table, const int32_t* seq_lens, void* stream);

/*
 * Scoring step alone: query folding/quantisation and the exact int32 scores, reduced to
 * one maximum per 16-token block. block_max: int32 [batch][hkv][max_pages_per_seq];
 * entries of blocks that hold a candidate token are written, all others are left
 * untouched. tile_max (nullable): int32 [batch][hkv][ceil(max_pages_per_seq / 4)], the
 * maximum of each 64-token tile's candidate tokens (tile c = tokens [64c, 64c + 64)),
 * written for tiles holding a candidate token; with 64-token chunks it is the module-1
 * chunk score. (HCAttention: global approximate scoring over quantised keys.)
 */
int32_t hsa_score_blocks(const hsa_dims* d, const void* q, const int8_t* kq,
                         const float* k_scale, const int32_t* page_table,
                         const int32_t* seq_lens, int32_t* block_max, int32_t* tile_max,
                         void* stream);

/*
 * The two pruning modules on precomputed block maxima (InfiniteHiP article, section
 * "实现 7.24 倍的端到端解码加速"). tile_max (nullable) as written by hsa_score_blocks; with
 * d->chunk == 64 it may be read instead of reducing block_max (the two must agree).
 * block_max and tile_max must be 16-byte aligned (else HSA_ERR_INVALID_ARG). chunk_idx
 * int32 [batch][hkv][k1] (nullable), n_chunks int32 [batch][hkv] (nullable), block_idx
 * int32 [batch][hkv][k2], n_blocks int32 [batch][hkv]. Limit: at most 53248 chunks per
 * sequence (ceil(max_pages_per_seq * 16 / chunk)); larger returns HSA_ERR_UNSUPPORTED.
 */
int32_t hsa_prune(const hsa_dims* d, const int32_t* seq_lens, const int32_t* block_max,
                  const int32_t* tile_max, int32_t* chunk_idx, int32_t* n_chunks,
                  int32_t* block_idx, int32_t* n_blocks, void* stream);

/*
 * hsa_score_blocks followed by hsa_prune, with the block maxima kept in the
 * HSA_OP_SELECT workspace. chunk_idx and n_chunks are nullable.
 */
int32_t hsa_select(const hsa_dims* d, const void* q, const int8_t* kq, const float* k_scale,
                   const int32_t* page_table, const int32_t* seq_lens, int32_t* chunk_idx,
                   int32_t* n_chunks, int32_t* block_idx, int32_t* n_blocks, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Sparse decode attention over T_b ("KV Cache 与长上下文推理", section "KV Cache 回顾":
 * softmax(q K^T / sqrt(d_k)) V, restricted to T_b). block_idx / n_blocks as produced by
 * hsa_select (entries outside [0, n_blocks) are ignored; kept blocks are clipped to
 * C_b). out: f32 [batch][hq][128]; lse: f32 [batch][hq] (natural log of the softmax
 * denominator of the scaled logits; nullable). With d->kv_on_host the K/V pages are read
 * from pinned host memory, only for the attended blocks (HCAttention: values stay in
 * CPU memory and are fetched late; InfiniteHiP article, latency section: the attention
 * kernel reads CPU memory while it runs).
 */
int32_t hsa_attend(const hsa_dims* d, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* page_table, const int32_t* seq_lens, const int32_t* block_idx,
                   const int32_t* n_blocks, float* out, float* lse, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Dense decode attention over every token [0, N_b): the in-run comparison point (same
 * kernels as hsa_attend with every block attended). Arguments as hsa_attend.
 */
int32_t dense_decode(const hsa_dims* d, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* page_table, const int32_t* seq_lens, float* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Inputs and outputs of one whole decode step. */
typedef struct hsa_step_io {
  const void* q;      /* bf16 [batch][hq][128] */
  const void* k_new;  /* bf16 [batch][hkv][128]: the new token's key */
  const void* v_new;  /* bf16 [batch][hkv][128]: the new token's value */
  float* out;         /* f32 [batch][hq][128] */
  float* lse;         /* f32 [batch][hq] (nullable) */
  int32_t io_on_host; /* 1: the five pointers above are PINNED HOST memory. When the device
                         addresses all of it (it reads host memory through the host's page
                         tables, or cudaHostGetDevicePointer succeeds: the default for pinned
                         memory with unified addressing), a kernel reads the inputs and the
                         attention writes the outputs over the host link; otherwise the call
                         copies the inputs in and the outputs back with cudaMemcpyAsync.
                         Either way everything is ordered on `stream`: the caller
                         synchronises it before reading the outputs or reusing the inputs. */
} hsa_step_io;

/*
 * One whole decode step: hsa_append_kv, hsa_select, hsa_attend on `stream`. seq_lens
 * already count the new token. block_idx / n_blocks receive the selection (device,
 * nullable: then the HSA_OP_STEP workspace holds it). Needs HSA_OP_STEP workspace.
 * The kernels read every input from its buffer when they run, so the first call with a
 * given set of argument values (the dims, the io struct's fields, every pointer, the
 * workspace size, the current device) records its launches into a CUDA graph, and later
 * calls with the same values launch that graph on `stream`: one launch a step in a decode
 * loop. The 64 most recently used sets are kept (CUDA driver resources, never freed before
 * exit). Calls on a stream that is being captured, or with the environment variable
 * HSA_STEP_GRAPHS=0, launch the kernels one by one. Results are the same either way.
 */
int32_t hsa_decode_step(const hsa_dims* d, const hsa_step_io* io, void* k_cache, void* v_cache,
                        int8_t* kq, const float* k_scale, const int32_t* page_table,
                        const int32_t* seq_lens, int32_t* block_idx, int32_t* n_blocks,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * A decode step that reuses an earlier step's selection (InfiniteHiP article, section
 * "实现 7.24 倍的端到端解码加速": the pruning result is kept for several decode steps and
 * refreshed every few): hsa_append_kv, then hsa_attend over the sink, the window and the
 * kept blocks block_idx / n_blocks (device inputs, as written by a previous hsa_decode_step;
 * required when k2 > 0), each clipped to the current candidate region [sink, N - window).
 * No scoring and no pruning. Same io, workspace (HSA_OP_STEP) and errors as hsa_decode_step.
 */
int32_t hsa_decode_step_reuse(const hsa_dims* d, const hsa_step_io* io, void* k_cache,
                              void* v_cache, int8_t* kq, const float* k_scale,
                              const int32_t* page_table, const int32_t* seq_lens,
                              const int32_t* block_idx, const int32_t* n_blocks, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * GPU block cache in front of K/V in host memory (InfiniteHiP article, section "实现 7.24 倍
 * 的端到端解码加速": the GPU keeps a cache of recently used KV blocks with an LRU policy and
 * the rest stays in host memory). One caller-owned device buffer of hsa_block_cache_bytes
 * bytes, 256-byte aligned and zero-filled before its first use, holds up to `capacity`
 * (page, kv head) blocks of bf16 K and V (8 KiB each) and their bookkeeping; it belongs to
 * one descriptor's cache (same num_pages, hkv) and must not be used by two calls that may
 * overlap on the GPU. capacity: at least batch * hkv * (ceil(sink / 16) + ceil(window / 16)
 * + 1 + k2) (one call's blocks) and at most 32768; otherwise hsa_block_cache_bytes returns 0
 * and the calls HSA_ERR_INVALID_ARG / HSA_ERR_UNSUPPORTED.
 *
 * Each call: its blocks (sink pages, window pages, kept blocks of every sequence and kv head)
 * are looked up; a hit counts as a use; every miss takes a slot among those this call does
 * not use and is copied in over the host link; the page that holds each sequence's last token
 * is copied again on every call (the append writes it). The host K/V of pages held in the
 * cache must not change otherwise. Two sequences may not share a page (reported as
 * HSA_ERR_DEVICE_CHECK through the error word). The victims, taken in ascending slot order by
 * the misses in call order, are the free slots (lower slot first), then:
 *  - d->cache_policy 0: the slots used longest ago (ties: the lower slot);
 *  - d->cache_policy 1 (HCAttention excerpt, contribution list: dynamic, reversible eviction
 *    of the least important KV pairs from the GPU cache by a cumulative-magnitude
 *    criterion): the slots whose blocks have the least cumulative attention mass (ties: the
 *    lower slot). The buffer keeps, for every (page, kv head) block, the sum over calls of the
 *    softmax probability that the block's attended tokens received from the kv head's query
 *    heads (fp32, zero until the block is first attended); each cached call adds its own.
 *    An evicted block keeps its sum and stays in host memory, so it returns when selected.
 *    hsa_block_cache_mass reads the sums. Needs at most 8192 segments per (sequence, kv
 *    head), ceil(sink / 16) + ceil(window / 16) + 1 + k2 <= 8192 (else UNSUPPORTED), and
 *    distinct block ids in each block_idx row (as hsa_prune writes them).
 */
size_t hsa_block_cache_bytes(const hsa_dims* d, int32_t capacity);

/*
 * Device pointer to the block cache's cumulative attention masses inside `block_cache`:
 * float [num_pages][hkv], entry page * hkv + h for (page, kv head h), updated by the cached
 * calls under cache_policy 1 (left at zero under policy 0). NULL if d or capacity is invalid.
 */
float* hsa_block_cache_mass(const hsa_dims* d, void* block_cache, int32_t capacity);

/*
 * hsa_attend for K/V in pinned host memory (d->kv_on_host = 1, mapped) through the block
 * cache: the attention itself reads the cached copies in device memory. Needs the
 * HSA_OP_CACHED workspace. Results equal hsa_attend's within floating-point rounding.
 */
int32_t hsa_attend_cached(const hsa_dims* d, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* page_table,
                          const int32_t* seq_lens, const int32_t* block_idx,
                          const int32_t* n_blocks, void* block_cache, int32_t capacity,
                          float* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * hsa_decode_step for K/V in pinned host memory with its attention through the block cache
 * (see hsa_attend_cached). Needs the HSA_OP_STEP workspace.
 */
int32_t hsa_decode_step_cached(const hsa_dims* d, const hsa_step_io* io, void* k_cache,
                               void* v_cache, int8_t* kq, const float* k_scale,
                               const int32_t* page_table, const int32_t* seq_lens,
                               int32_t* block_idx, int32_t* n_blocks, void* block_cache,
                               int32_t capacity, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * hsa_select without a workspace, for callers that cannot allocate device memory: code
 * embedded in a host program that owns every device allocation through its own pool, or
 * that runs on a latency-critical path where cudaMalloc (which can synchronise the device)
 * is not allowed. Nothing in the method calls for this; the pages have no counterpart.
 * Same arguments and results as hsa_select minus the workspace. Its scratch (a device error
 * word, then the block and tile score maxima) is one fixed 4 MiB device array inside the
 * library, held by every GPU that loads the library until the process exits: shapes with
 *   256 + round256(4 * batch * rows * max_pages_per_seq)
 *       + round256(4 * batch * rows * ceil(max_pages_per_seq / 4)) > 4 MiB,
 * rows = hq with per-head selection (d->per_head = 1), else hkv (e.g. more than about 800K
 * 16-token blocks summed over sequences and kv heads, G times fewer with per-head
 * selection), return HSA_ERR_WORKSPACE_TOO_SMALL. The first call on a device loads the
 * library's device code there (make it before any stream capture); every call looks the
 * array's device address up in the current context. All calls share the array and it keeps
 * the last call's contents (each call writes every maximum it then reads, so only the error
 * word must start at zero, which it does); calls that may overlap on the GPU, on any
 * stream, race on it and must be ordered by the caller. Device-side failures (a bounds
 * check, or a bounded wait that ran out, after which the selection may be stale) set the
 * array's error word: read and clear it with hsa_read_device_error(NULL, stream, &code).
 * Calls no allocating routine.
 */
int32_t hsa_select_noalloc(const hsa_dims* d, const void* q, const int8_t* kq,
                           const float* k_scale, const int32_t* page_table,
                           const int32_t* seq_lens, int32_t* chunk_idx, int32_t* n_chunks,
                           int32_t* block_idx, int32_t* n_blocks, void* stream);

/*
 * The number of kernels hsa_decode_step launches for d with device-memory inputs and a
 * 16-byte-aligned page table: 2 when the sparse attention runs the pruning modules itself
 * (64-token chunks, two modules, rows of up to 2048 chunk scores for 8 query heads a kv
 * head or 2304 otherwise, K/V in device memory) and the scorer appends the new token
 * (window >= 1), 3 with no window (the append first), else 4 (scorer, append, pruning
 * kernel, attention). Host I/O adds a staging kernel. -1 for an invalid d.
 */
int32_t hsa_decode_step_kernels(const hsa_dims* d);

/*
 * Reads and clears the device error word of `workspace` after synchronising `stream`:
 * *code receives HSA_OK, HSA_ERR_TIMEOUT or HSA_ERR_DEVICE_CHECK. workspace NULL: the error
 * word of hsa_select_noalloc's fixed scratch array on the current device. This is the one
 * call that synchronises.
 */
int32_t hsa_read_device_error(void* workspace, void* stream, int32_t* code);

#ifdef __cplusplus
}
#endif

#endif /* HSA_H_ */
