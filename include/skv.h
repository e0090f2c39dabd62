/*
 * skv.h -- C ABI of the GB300 speculative-KV-coding library (libskv.so).
 *
 * Lossless coding of a target model's KV cache against a predictor's
 * approximation of it.  Sources (page title, section):
 *   [SKV]  "Speculative KV coding: losslessly compressing KV cache by up to ~4x"
 *          (summary at aisparkup.com/posts/13411), sections "core idea" and
 *          "which predictor".
 *   [DCKV] "DCKV compresses a hybrid language model's prompt KV cache with
 *          learned transform coding" (onedev.kr/papers/1428), sections "how it
 *          works", "how it differs" and "usage".
 *
 * Conventions for every call:
 *   - Pointers prefixed d_ are device memory owned by the caller; h_ pointers
 *     are host memory.  The library allocates nothing and frees nothing.
 *   - Device buffers must be 16-byte aligned (cudaMalloc gives 256), and a
 *     bitstream buffer must be readable up to the next multiple of 16 bytes
 *     past its end (the decoder reads whole aligned 16-byte blocks).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue their kernels on it and return without waiting,
 *     except where a call says it synchronises.
 *   - Argument errors are reported synchronously (SKV_ERR_INVALID_ARG or
 *     SKV_ERR_UNSUPPORTED) before anything is launched.  Launch failures give
 *     SKV_ERR_CUDA.  Errors found by kernels while they run (a corrupt stream,
 *     too small an output buffer, an out-of-range bin) are recorded in a
 *     caller-owned 32-bit device status word and read with skv_read_status.
 *   - Kernels never trap; a bad stream gives a status, never a fault.
 *
 * Data layouts:
 *   KV cache (FP8 E4M3 or BF16 bit patterns): [layer][kv][head][token][head_dim],
 *     row-major.  Channel c = ((layer*n_kv + kv)*n_heads + head)*head_dim + d.
 *   Coefficient stream (COEF): q int16 [token][coef], row-major; means mu fp32
 *     [token][coef] (in quantisation-step units); scales beta fp32 [coef].
 *
 * Stream format (what the oracle reproduces byte for byte):
 *   A slice is one (layer, kv, head) block of n_tokens*head_dim positions
 *   (COEF: the whole [token][coef] grid).  Each slice is cut into chunks of
 *   32*lane_syms positions (the last one may be short).  Positions come in
 *   groups of 16 bytes (16 FP8 values, 8 BF16 or COEF values); lane l of a
 *   chunk owns the groups whose chunk-local index is l mod 32.  Each lane is an
 *   independent rANS stream with a 32-bit state in [2^16, 2^32), 16-bit
 *   renormalisation and 12-bit probabilities ([DCKV] how it differs: GPU rANS
 *   over Laplace-integrated probabilities), coded backwards:
 *     lane words (u16, little endian) = [x_final >> 16, x_final & 0xFFFF,
 *                                        renormalisation words, last first]
 *   Symbols: residual r = ord(target) - ord(pred) of monotone ordinals
 *   ([SKV] core idea); |r| <= 127 -> symbol r + 127, otherwise the escape
 *   symbol 255 followed by the residual mod 2^width as raw bytes (uniform
 *   steps of frequency 16, high byte decoded first).  COEF: r = q - floor(mu'),
 *   mu' = mu rounded to 1/16, and components with beta < 0.05 carry no
 *   symbols ([DCKV] how it works) and decode to 0.
 *   Lanes are stored in lane order (chunk*32 + l); lane_offsets[g] is the
 *   byte offset of lane g and lane_offsets[n_lanes] the total size.
 */
#ifndef SKV_H
#define SKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKV_PARAMS_VERSION 1u

/* status codes */
#define SKV_OK 0
#define SKV_ERR_INVALID_ARG 1
#define SKV_ERR_CUDA 2
#define SKV_ERR_CAPACITY 3
#define SKV_ERR_CORRUPT 4
#define SKV_ERR_TIMEOUT 5
#define SKV_ERR_UNSUPPORTED 6

/* dtype codes */
#define SKV_FP8_E4M3 1u
#define SKV_BF16 2u
#define SKV_COEF_I16 3u

/* Table blob: table t occupies SKV_TABLE_STRIDE bytes at t*SKV_TABLE_STRIDE.
 * Within a table:
 *   SKV_TABLE_ENC_OFF  256 x {u32 m_lo, u32 w}: encoder entries with
 *                      w = fr << 20 | cum << 8 | 1 << 7 | s, s = ceil(log2 fr),
 *                      where m = 2^32 + m_lo = ceil(2^(32+s) / fr) and
 *                      floor(x / fr) = (umulhi(x, m_lo) + x) >> s
 *                      exactly for every state x < fr*2^20 the encoder meets
 *   SKV_TABLE_LUT_OFF  4096 x u8: symbol owning each 12-bit slot
 *   SKV_TABLE_DEC_OFF  256 x u32: fr | (-cum mod 2^16) << 16 (the upper half
 *                      read as a signed 16-bit number is -cum)
 *   SKV_TABLE_FREQ_OFF 256 x u16: frequencies (sum 4096, each >= 1)
 *   SKV_TABLE_CUM_OFF  257 x u16: cumulative frequencies (cum[256] = 4096)
 * KV streams have 32 tables (scale bin b = table b); COEF streams have 1024
 * (table 16*b + f: scale bin b, mean fraction f/16).  A COEF blob continues,
 * at n_tables * SKV_TABLE_STRIDE, with SKV_TABLE_SLOT_BYTES per table: 4096 x
 * u32 slot entries sym | fr << 8 | (slot - cum) << 20 (the slot's symbol, its
 * frequency and the slot's offset within it: one read per decoding step for
 * tables that stay in L2).  skv_tables_bytes gives the whole blob's size. */
#define SKV_TABLE_STRIDE 8704u
#define SKV_TABLE_SLOT_BYTES 16384u
#define SKV_TABLE_ENC_OFF 0u
#define SKV_TABLE_LUT_OFF 2048u
#define SKV_TABLE_DEC_OFF 6144u
#define SKV_TABLE_FREQ_OFF 7168u
#define SKV_TABLE_CUM_OFF 7680u

/* Status-word bits set by kernels (skv_read_status maps them to codes). */
#define SKV_FLAG_CORRUPT 1u
#define SKV_FLAG_CAPACITY 2u
#define SKV_FLAG_TIMEOUT 4u
#define SKV_FLAG_BAD_BIN 8u
#define SKV_FLAG_BAD_BLOCK 16u

typedef struct {
  uint32_t version;   /* SKV_PARAMS_VERSION                                     */
  uint32_t dtype;     /* SKV_FP8_E4M3, SKV_BF16 or SKV_COEF_I16                 */
  uint32_t n_layers;  /* KV only                                                */
  uint32_t n_kv;      /* KV only: 2 for {K, V}                                  */
  uint32_t n_heads;   /* KV only: KV heads                                      */
  uint32_t head_dim;  /* KV only: multiple of 16 (FP8) / 8 (BF16) dividing 512 / 256 */
  uint64_t n_tokens;
  uint32_t n_coef;    /* COEF only: coefficients per token                      */
  uint32_t lane_syms; /* positions per lane (chunk = 32 lanes); a multiple of
                         the group size (16 FP8, 8 otherwise), at most 65536    */
  uint32_t n_calib;   /* KV only: calibration tokens per channel (<= 65536)     */
  uint32_t model;     /* residual model: 0 = one Laplace scale bin per channel;
                         1 (FP8 only) = the channel's scale normalised by the
                         prediction's exponent (see SKV_MODEL_EXPONENT)        */
} skv_params;

/* Residual models ([SKV] names more refined residual models as the next
 * step; the plain reading below is this library's).
 * SKV_MODEL_CHANNEL: calibration stores per channel the bin (0..31) of the
 *   Laplace scale fitted on |r|, and every position uses that table.
 * SKV_MODEL_EXPONENT (FP8): ordinals are evenly spaced in bit patterns, so
 *   one value-space error spans half as many ordinals per step up of the
 *   prediction's exponent field e = (pred_bits >> 3) & 15.  Calibration fits
 *   the scale on |r| * 2^e (S_c = sum of |r| 2^e, q = floor(S_c 2^16 / N))
 *   and stores its base bin on the scale grid extended upward (4 bins per
 *   octave, 0 below 1/8, no cap); a position then uses table
 *   min(max(base - 4 e, 0), 31).  d_sum_abs receives S_c (saturated at
 *   2^32 - 1). */
#define SKV_MODEL_CHANNEL 0u
#define SKV_MODEL_EXPONENT 1u

/* Text for a status code (static storage). */
const char* skv_status_string(int status);

/* SKV_OK if the parameters describe a supported stream, else
 * SKV_ERR_INVALID_ARG / SKV_ERR_UNSUPPORTED.  Host only. */
int skv_check_params(const skv_params* p);

/* Sizes (host only; 0 for invalid parameters). */
uint64_t skv_num_positions(const skv_params* p); /* values in the target          */
uint64_t skv_num_channels(const skv_params* p);  /* entries of the bins array      */
uint32_t skv_num_tables(const skv_params* p);    /* 32 (KV) or 1024 (COEF)         */
uint64_t skv_num_chunks(const skv_params* p);
uint64_t skv_num_lanes(const skv_params* p);     /* lane_offsets has n_lanes + 1   */
uint64_t skv_tables_bytes(const skv_params* p);  /* num_tables * SKV_TABLE_STRIDE (+ slot entries, COEF) */
uint64_t skv_max_bitstream_bytes(const skv_params* p); /* worst case of any input  */
uint64_t skv_encode_workspace_bytes(const skv_params* p);

/* Calibration ([SKV] which predictor: residual statistics measured once on a
 * small calibration set, then frozen; [DCKV] how it differs: a per-component
 * Laplace).  KV: for every channel, S = sum of |ord(target) - ord(pred)| over
 * tokens [0, min(n_calib, n_tokens)); the Laplace scale estimate S/N (Q16,
 * floored) selects one of 32 scale bins (4 per octave over [1/8, 32), clamped).
 * Writes d_bins[n_channels].  d_sum_abs[n_channels] (u32 S) and
 * d_hist[n_channels][256] (u32 symbol counts of the calibration tokens) are
 * optional (NULL to skip); d_hist is accumulated, so the caller zeroes it.
 * COEF: d_target is ignored (may be NULL), d_pred is beta[n_coef] fp32
 * (scale / step); bins are 0xFF for beta < 0.05 (switched off, [DCKV] how it
 * works) or one of 64 bins (8 per octave); d_sum_abs and d_hist must be NULL. */
int skv_calibrate(const skv_params* p, const void* d_target, const void* d_pred,
                  uint8_t* d_bins, uint32_t* d_sum_abs, uint32_t* d_hist, void* stream);

/* Builds every probability table of the stream into d_tables
 * (skv_tables_bytes(p) bytes): Laplace masses integrated over integer cells
 * ([DCKV] how it differs) from exact integer arithmetic, quantised to
 * frequencies summing to 4096 with a floor of 1.  Depends only on p's dtype. */
int skv_build_tables(const skv_params* p, void* d_tables, uint64_t tables_bytes, void* stream);

/* Encode ([SKV] core idea, steps 1-2).  Inputs: d_target and d_pred caches
 * (COEF: d_target = q int16, d_pred = mu fp32), tables from skv_build_tables
 * and bins from skv_calibrate.  Outputs: d_bitstream (cap_bytes available)
 * and d_lane_offsets[n_lanes + 1] (u64 byte offsets).  d_workspace must hold
 * skv_encode_workspace_bytes(p) bytes.  d_status (one u32) is cleared and then
 * collects kernel flags.  If h_total_bytes is non-NULL the call synchronises
 * the stream once, stores the stream size there and returns SKV_ERR_CAPACITY
 * if it exceeds cap_bytes (the bitstream is then not written); if NULL the call
 * is fully asynchronous and an overflow sets SKV_FLAG_CAPACITY. */
int skv_encode(const skv_params* p, const void* d_target, const void* d_pred,
               const void* d_tables, const uint8_t* d_bins, void* d_bitstream,
               uint64_t cap_bytes, uint64_t* d_lane_offsets, void* d_workspace,
               uint64_t workspace_bytes, uint32_t* d_status, uint64_t* h_total_bytes,
               void* stream);

/* Decode ([SKV] core idea, steps 3-4: the decoder re-uses the same prediction
 * and adds the decoded residual back).  Writes the exact target bits into
 * d_target_out (COEF: q int16; switched-off components are 0).  A lane whose
 * stream does not end in the initial state or does not consume exactly its
 * words, or offsets that are not increasing and inside n_bytes, set
 * SKV_FLAG_CORRUPT in d_status (cleared by the call first).  The decoder reads
 * the stream in aligned 16-byte blocks: d_bitstream must be readable up to
 * n_bytes rounded up to a multiple of 16 (the bytes past n_bytes are ignored). */
int skv_decode(const skv_params* p, const void* d_bitstream, uint64_t n_bytes,
               const uint64_t* d_lane_offsets, const void* d_pred, const void* d_tables,
               const uint8_t* d_bins, void* d_target_out, uint32_t* d_status, void* stream);

/* Paged KV caches (block pools, as serving systems keep them; [SKV] core idea
 * for prefill-to-decode transfer and prefix caches).  The pages define no
 * layout; this one keeps each token's heads and channels together:
 *   pool (l, kv) of every layer l and K/V index kv holds n_blocks blocks;
 *   block b holds block_tokens consecutive tokens as [block_tokens][n_heads]
 *   [head_dim] (row-major); the pools are contiguous, pool (l, kv) first,
 *   so element (l, kv, b, row, h, d) sits at index
 *   ((((l * n_kv + kv) * n_blocks + b) * block_tokens + row) * n_heads + h)
 *   * head_dim + d of d_*_pool (elements of 1 byte for FP8, 2 for BF16).
 * d_block_table[j] (u32, j < ceil(n_tokens / block_tokens)) is the block that
 * holds tokens [j * block_tokens, (j + 1) * block_tokens) in every pool; rows
 * past n_tokens in the last block are not read or written.  block_tokens must
 * be a power of two.  The caller owns the pools and the table.
 *
 * The paged calls compute exactly what the dense calls compute on the cache
 * gathered into [layer][kv][head][token][head_dim]: the same bins, the same
 * bitstream and lane offsets, and a decode that writes the target bits into
 * the target pool's rows (other rows untouched).  KV dtypes only (COEF streams:
 * SKV_ERR_UNSUPPORTED).  A block-table entry >= n_blocks sets
 * SKV_FLAG_BAD_BLOCK in d_status (skv_read_status: SKV_ERR_INVALID_ARG); its
 * rows are then read from block 0 and never written. */
typedef struct {
  const uint32_t* d_block_table;
  uint32_t n_blocks;     /* blocks per (layer, K/V) pool */
  uint32_t block_tokens; /* tokens per block, a power of two */
} skv_paged_layout;

/* skv_calibrate on paged pools; d_status (one u32, cleared first) collects
 * SKV_FLAG_BAD_BLOCK. */
int skv_calibrate_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_target_pool,
                        const void* d_pred_pool, uint8_t* d_bins, uint32_t* d_sum_abs, uint32_t* d_hist,
                        uint32_t* d_status, void* stream);

/* skv_encode on paged pools (same workspace, outputs and status rules). */
int skv_encode_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_target_pool,
                     const void* d_pred_pool, const void* d_tables, const uint8_t* d_bins, void* d_bitstream,
                     uint64_t cap_bytes, uint64_t* d_lane_offsets, void* d_workspace, uint64_t workspace_bytes,
                     uint32_t* d_status, uint64_t* h_total_bytes, void* stream);

/* skv_decode into the rows of a paged target pool. */
int skv_decode_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_bitstream,
                     uint64_t n_bytes, const uint64_t* d_lane_offsets, const void* d_pred_pool,
                     const void* d_tables, const uint8_t* d_bins, void* d_target_pool_out, uint32_t* d_status,
                     void* stream);

/* Checkerboard context for coefficient streams ([DCKV] how it differs: the
 * compressed rows are split by token parity; even rows are coded with the
 * token-conditioned means alone, odd rows with means that also use the
 * already decoded rows on both sides through a rank-1024 linear map, so each
 * parity decodes in one token-parallel pass).  The page's map is learned; this
 * call takes any integer map of the same shape (the caller's, e.g. a seeded
 * one) and computes, for odd row t (token 2t + 1),
 *   x   = clamp(q_even[t] + q_even[t + 1], -127, 127)   (no row t+1: 0)
 *   g_r = clamp(floor((V x)_r / 2^shift1), -127, 127)
 *   k_c = floor((U g)_c / 2^shift2)                     (1/16 steps)
 *   mu' = clamp(mu_q + k, -(2^23 - 1), 2^23 - 1) / 16
 * with V, U entries used clamped to [-8, 8] and mu_q = floor(16 mu + 1/2) the
 * coefficient mean quantisation of d_mu_odd (the token-conditioned means of
 * the odd rows).  mu' is exact in fp32 and quantises back to mu_q + k, so the
 * odd rows are an ordinary COEF stream (skv_encode / skv_decode with n_tokens
 * = n_odd and d_pred = mu'), coded after (and decoded after) the even rows'
 * stream (n_tokens = n_even, d_pred = their means).
 * Rows are [row][n_coef] (q int16, means fp32); n_odd <= n_even, n_odd below
 * 8388480.  Both products run on the 5th-generation tensor cores (tcgen05,
 * bf16 operands, fp32 accumulators in tensor memory) and are exact (small
 * integers, fp32 sums below 2^24).  n_coef and rank: multiples of 32 up to
 * 16384; shifts <= 30.
 * d_scratch: skv_ctx_scratch_bytes(n_odd, n_coef, rank) bytes, 16-aligned
 * (x and g as bf16 matrices and bf16 copies of V and U).
 * d_status: one caller-owned device word, cleared by the call; a kernel that
 * waited over about a second on its own pipeline sets SKV_FLAG_TIMEOUT
 * (read it with skv_read_status); its output tile is then not written
 * (d_mu_out is undefined after a timeout).  Argument errors return
 * SKV_ERR_INVALID_ARG and launch nothing; SKV_ERR_UNSUPPORTED if the driver
 * offers no tensor-map encoder. */
typedef struct {
  const int8_t* d_V;   /* [rank][n_coef] */
  const int8_t* d_U;   /* [n_coef][rank] */
  uint32_t rank;
  uint32_t shift1, shift2;
} skv_ctx_map;
uint64_t skv_ctx_scratch_bytes(uint64_t n_odd, uint32_t n_coef, uint32_t rank);
int skv_ctx_means(const skv_ctx_map* map, const int16_t* d_q_even, uint64_t n_even, const float* d_mu_odd,
                  uint64_t n_odd, uint32_t n_coef, float* d_mu_out, void* d_scratch, uint64_t scratch_bytes,
                  uint32_t* d_status, void* stream);

/* Host-resident caches ([SKV] core idea: the coded cache is what moves between
 * machines or sits in a prefix store; [VeriCache] "operational
 * considerations": a full KV cache that lives in host memory crosses the host
 * link, so the codec runs alongside the copies).  The target and prediction
 * caches (and, for decoding, the stream and its lane offsets) are in host
 * memory; page-locked memory (cudaHostAlloc / cudaMallocHost) lets the copies
 * overlap the kernels, pageable memory works but serialises them.  KV dtypes
 * only (COEF: SKV_ERR_UNSUPPORTED).
 *
 * The cache is coded in groups of group_layers layers (a layer range is an
 * independent sub-cache: chunks never straddle a slice, calibration is per
 * channel, tables depend only on the dtype), double-buffered in d_workspace
 * (skv_host_workspace_bytes(p, group_layers, group_cap_bytes) bytes, 16-byte
 * aligned, caller-owned): while group k is calibrated and coded on streams[1],
 * group k + 1 is copied in on streams[0] and group k - 1 copied out on
 * streams[2] (three caller-owned cudaStream_t).  group_cap_bytes bounds one
 * group's stream on the device (0: the group's worst case); a group that needs
 * more fails with SKV_ERR_CAPACITY.  Both calls are synchronous: they return
 * when every copy has landed, with the most serious status of any group (the
 * kernels' flags included).  They create and destroy a few CUDA events but
 * allocate no memory.
 *
 * skv_encode_host: calibrates every group into d_bins (n_channels, device,
 * written in full), encodes it with d_tables (from skv_build_tables) and writes
 * the stream to h_bitstream (cap_bytes) and the whole-cache lane offsets to
 * h_lane_offsets[n_lanes + 1]: the result is byte-identical to skv_calibrate +
 * skv_encode of the whole cache on the device.  *h_total_bytes (if non-NULL)
 * receives the stream size.  The device computes each group's place in the
 * stream; the host reads it from the offsets copied back, one group behind,
 * so the coding stream never waits on the host.
 *
 * skv_decode_host: decodes the stream (h_bitstream, n_bytes, h_lane_offsets)
 * against the prediction h_pred with d_tables and d_bins into h_target_out
 * (the cache's size).  Offsets that are not increasing or not inside n_bytes
 * give SKV_ERR_CORRUPT before anything is launched. */
uint64_t skv_host_workspace_bytes(const skv_params* p, uint32_t group_layers, uint64_t group_cap_bytes);
int skv_encode_host(const skv_params* p, const void* h_target, const void* h_pred, const void* d_tables,
                    uint8_t* d_bins, void* h_bitstream, uint64_t cap_bytes, uint64_t* h_lane_offsets,
                    uint64_t* h_total_bytes, uint32_t group_layers, uint64_t group_cap_bytes, void* d_workspace,
                    uint64_t workspace_bytes, void* const* streams);
int skv_decode_host(const skv_params* p, const void* h_bitstream, uint64_t n_bytes, const uint64_t* h_lane_offsets,
                    const void* h_pred, const void* d_tables, const uint8_t* d_bins, void* h_target_out,
                    uint32_t group_layers, uint64_t group_cap_bytes, void* d_workspace, uint64_t workspace_bytes,
                    void* const* streams);

/* Encode without a caller-provided workspace.  The pages have no counterpart
 * to this call; it exists for callers that cannot allocate device memory, such
 * as code handed only its input and output buffers by a host framework that
 * owns every allocation, or code running where the device's memory has already
 * been claimed by another pool and a cudaMalloc would fail.
 *
 * Same arguments and results as skv_encode minus the workspace.  The scratch
 * is a file-scope device array of SKV_NOALLOC_SCRATCH_BYTES (64 MiB) inside
 * libskv.so, which every GPU that loads the library holds until the process
 * exits.  A stream fits when skv_encode_workspace_bytes(p) is at most that
 * size: about 8.3 million FP8 positions (254 chunks at lane_syms 1024, 63 at
 * 4096) or 5.5 million BF16 positions (170 chunks at lane_syms 1024); larger
 * streams are rejected with SKV_ERR_UNSUPPORTED before anything is launched.
 *
 * The first call on a device looks up the array's device address on the
 * current device (once per device, then cached); make that first call before
 * any stream capture.  The call itself allocates nothing and frees nothing.
 * Every call on a device shares the one array and it keeps the last call's
 * contents: the call clears the per-chunk look-back states and the chunk
 * ticket itself, and every other scratch word is written before it is read.
 * Calls whose work overlaps on the GPU (different streams, or other host
 * threads) race on the array: serialise them. */
#define SKV_NOALLOC_SCRATCH_BYTES (64ull << 20)
int skv_encode_noalloc(const skv_params* p, const void* d_target, const void* d_pred,
                       const void* d_tables, const uint8_t* d_bins, void* d_bitstream,
                       uint64_t cap_bytes, uint64_t* d_lane_offsets, uint32_t* d_status,
                       uint64_t* h_total_bytes, void* stream);

/* Self-test of the encoder's bounded wait (no counterpart on the pages): runs
 * the encoder's chunk look-back for chunks 0..n_chunks-1 (chunk w has w + 1
 * bytes) on d_state[n_chunks] (u64, cleared by the call), except that chunk
 * missing_chunk never publishes.  Chunks before it receive their exclusive
 * prefix in d_excl[w]; the chunk after it must give up after max_spins polls
 * (about 100 ns each), set SKV_FLAG_TIMEOUT in d_status and mark itself
 * failed, and every later chunk must fail at once (d_excl = ~0).  At most 4096
 * chunks (all resident); nothing waits without a limit. */
int skv_selftest_lookback(uint64_t* d_state, uint32_t n_chunks, uint32_t missing_chunk,
                          uint32_t max_spins, uint64_t* d_excl, uint32_t* d_status, void* stream);

/* Self-test of the bounded waits of the tensor-core context products (no
 * counterpart on the pages): launches one tile of the first product with its
 * tile loads switched off, so that the MMA thread's wait for operands runs out
 * after about a second; the kernel must then set SKV_FLAG_TIMEOUT in d_status,
 * free its tensor memory and return.  d_scratch: 48 KB, 16-byte aligned,
 * caller-owned (its contents are overwritten). */
int skv_selftest_ctx_wait(void* d_scratch, uint32_t* d_status, void* stream);

/* Checked build (no counterpart on the pages; it stands in for a memory
 * checker): a library compiled with -DSKV_CHECKED=1 checks every
 * shared-memory access of the codec kernels against the launch's shared size
 * and alignment, and the encoder's table, word-buffer and scratch-slot
 * cursors, the decoder's output rows, the chunk copy into the stream and the
 * coefficient table indices against their own regions.  A failed check is
 * counted, the first failing site is kept and the access is skipped; nothing
 * traps.  This call synchronises the device, returns the count and the first
 * site in *h_count / *h_first_site and clears both.  In the ordinary build it
 * returns SKV_ERR_UNSUPPORTED. */
int skv_checked_failures(uint32_t* h_count, uint32_t* h_first_site);

/* Synchronises the stream, reads the status word and returns SKV_OK or the
 * code of the most serious flag (CORRUPT > CAPACITY > TIMEOUT > INVALID_ARG
 * for an out-of-range bin or block-table entry). */
int skv_read_status(const uint32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H */
