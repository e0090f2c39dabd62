// skv.cu -- speculative KV coding on GB300 (sm_103a): kernels and the C ABI.
//
// Hot path: lossless coding of a target KV cache against a predictor's
// approximation of it ([SKV] "Speculative KV coding", section "core idea"):
// monotone ordinals, residual symbols with an escape, per-channel Laplace
// tables from calibration tokens ([SKV] "which predictor"; [DCKV] "how it
// differs": per-component Laplace integrated over quantisation cells, GPU
// rANS) and 32-lane interleaved rANS.  Page references:
//   [SKV]  "Speculative KV coding: losslessly compressing KV cache by up to ~4x"
//   [DCKV] "DCKV compresses a hybrid language model's prompt KV cache with
//          learned transform coding"
//
// Kernels.  The codec is integer work bound by the SM's integer and
// shared-memory pipes (HBM is the roofline); only the checkerboard context map
// is a dense contraction and runs on the tensor cores:
//   k_build_tables    one CTA per table: Q32 Taylor exp, power chain, masses,
//                     largest-remainder frequencies, encoder reciprocals,
//                     slot->symbol table (and, COEF, one-read slot entries)
//   k_calibrate_kv    one CTA per (layer, kv, head) slice: exact sum |r| per
//                     channel over the calibration tokens, warp reductions,
//                     optional histograms, scale bins
//   k_encode_kv       persistent warps taking chunks (32 lanes) from a ticket,
//                     128-bit coalesced loads of both caches (each lane owns
//                     16-byte groups), encoder tables in shared memory, reverse
//                     pass into per-lane shared-memory word buffers flushed to
//                     the warp's scratch slots; each chunk is placed in the
//                     stream by a decoupled look-back one chunk later
//   k_decode_kv       persistent warps, slot->symbol and decoder tables in
//                     shared memory, per-lane stream rings filled by cp.async,
//                     speculative FP8 groups, reconstruction fused in: ordinal
//                     of the prediction + residual, inverse ordinal, 128-bit
//                     stores
//   k_*_coef          transform-coefficient streams (1024 tables read through
//                     L1/L2; switched-off components carry no symbol), with
//                     k_scan_* (lane lengths -> byte offsets) and k_compact
//   k_ctx_*           checkerboard context: x rows and bf16 map factors, then
//                     two tcgen05 products (TMA-fed, accumulators in tensor
//                     memory)

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "skv.h"

namespace {

constexpr uint32_t kLanes = 32;
constexpr uint32_t kChain = 2056;        // tau^0 .. tau^2055 covers |16 s + 8 + 15| <= 2055
constexpr uint32_t kStateLow = 1u << 16; // rANS state lower bound L
constexpr uint32_t kKvTables = 32;
constexpr uint32_t kCoefTables = 1024;
// Shared-memory layout of the codec kernels.  Table strides are padded so
// that the same symbol of neighbouring tables falls in different banks:
// encoder entries are 8 bytes (stride/8 = 3 mod 16), decoder tables are the
// slot->symbol LUT followed by the 32-bit decoder entries (stride/4 = 5 mod 32).
// The skews are the ones with the fewest modelled bank conflicts on synthetic
// caches (symbols concentrated around the centre, four channel sets per
// half-warp in the encoder).
constexpr uint32_t kEncTabStride = 2048 + 24;
constexpr uint32_t kEncTabBytes = kKvTables * kEncTabStride;       // 66304
constexpr uint32_t kEmitBytes = 144;                               // per-lane word buffer
constexpr uint32_t kDecTabStride = 4096 + 1024 + 20;
constexpr uint32_t kDecTabBytes = kKvTables * kDecTabStride;       // 164480
constexpr uint32_t kRingBytes = 64;                                // per-lane stream ring
#ifndef SKV_RING_STRIDE
#define SKV_RING_STRIDE 64
#endif
constexpr uint32_t kRingStride = SKV_RING_STRIDE;   // spacing of the lanes' rings (16-byte multiple)
#ifndef SKV_CODEC_THREADS
#define SKV_CODEC_THREADS 1024
#endif
constexpr int kCodecThreads = SKV_CODEC_THREADS;   // decoder threads per CTA (one CTA per SM)
// the paged and exponent-model decoders keep more state per lane: 768 threads
// leave them enough registers not to spill
constexpr int dec_threads(bool paged, bool model) { return (paged || model) && kCodecThreads > 768 ? 768 : kCodecThreads; }
#ifndef SKV_ENC_THREADS
#define SKV_ENC_THREADS 768
#endif
constexpr int kEncThreads = SKV_ENC_THREADS;       // encoder threads per CTA (more registers per thread)
constexpr int kScanPerBlock = 4096;       // lanes per scan block (256 threads x 16)

// ---------------------------------------------------------------------------
// Host-side geometry
// ---------------------------------------------------------------------------
struct Geo {
  uint32_t dtype, esz, group, raw_bytes, K, D, C, n_tables, sub, model;
  uint64_t T, n_slices, slice_pos, cps, n_chunks, n_lanes, n_channels, n_positions;
  uint64_t slot_words;
};

int make_geo(const skv_params* p, Geo* g) {
  if (!p || !g) return SKV_ERR_INVALID_ARG;
  if (p->version != SKV_PARAMS_VERSION || p->model > SKV_MODEL_EXPONENT) return SKV_ERR_INVALID_ARG;
  if (p->model == SKV_MODEL_EXPONENT && p->dtype != SKV_FP8_E4M3) return SKV_ERR_UNSUPPORTED;
  memset(g, 0, sizeof(*g));
  g->dtype = p->dtype;
  g->model = p->model;
  if (p->dtype == SKV_FP8_E4M3) { g->esz = 1; g->group = 16; g->raw_bytes = 1; }
  else if (p->dtype == SKV_BF16) { g->esz = 2; g->group = 8; g->raw_bytes = 2; }
  else if (p->dtype == SKV_COEF_I16) { g->esz = 2; g->group = 8; g->raw_bytes = 2; }
  else return SKV_ERR_INVALID_ARG;
  g->K = p->lane_syms;
  if (g->K == 0 || g->K > 65536 || (g->K % g->group) != 0) return SKV_ERR_INVALID_ARG;
  g->T = p->n_tokens;
  if (g->T > (1ull << 40)) return SKV_ERR_UNSUPPORTED;
  if (p->dtype == SKV_COEF_I16) {
    if (p->n_coef == 0) return SKV_ERR_INVALID_ARG;
    g->C = p->n_coef;
    g->n_slices = 1;
    g->slice_pos = g->T * g->C;
    g->n_channels = g->C;
    g->n_tables = kCoefTables;
    g->sub = 8;
  } else {
    g->D = p->head_dim;
    if (g->D == 0 || (g->D % g->group) != 0 || ((32u * g->group) % g->D) != 0)
      return SKV_ERR_UNSUPPORTED;
    if (p->n_calib > 65536) return SKV_ERR_INVALID_ARG;
    g->n_slices = (uint64_t)p->n_layers * p->n_kv * p->n_heads;
    g->slice_pos = g->T * g->D;
    g->n_channels = g->n_slices * g->D;
    g->n_tables = kKvTables;
    g->sub = 4;
  }
  const uint64_t cs = (uint64_t)kLanes * g->K;
  g->cps = (g->slice_pos + cs - 1) / cs;
  g->n_chunks = g->n_slices * g->cps;
  g->n_lanes = g->n_chunks * kLanes;
  g->n_positions = g->n_slices * g->slice_pos;
  if (g->n_positions > (1ull << 44)) return SKV_ERR_UNSUPPORTED;
  // worst case per lane: 2 state words + one word per coding step, and an
  // escaped position takes 1 + raw_bytes steps; rounded to 16 bytes
  g->slot_words = ((2 + (uint64_t)g->K * (1 + g->raw_bytes)) + 7) & ~7ull;
  return SKV_OK;
}

uint64_t align256(uint64_t v) { return (v + 255) & ~255ull; }

// Upper bound on resident codec warps (152 SMs x 32 warps fit; larger devices
// are clamped to it).  KV encode scratch is one slot per lane of each warp.
constexpr uint64_t kMaxWarps = 5120;

struct WsLayout {
  uint64_t slots_off, lw_off, part_off, state_off, ticket_off, total;
  uint64_t n_scan_blocks, n_slots;
};

// KV: two sets of lane slots per warp (reused chunk after chunk) + chunk look-back states
// + the chunk ticket.  COEF: per-lane slots + lane lengths + scan partials.
WsLayout ws_layout(const Geo& g) {
  WsLayout w;
  memset(&w, 0, sizeof(w));
  if (g.dtype != SKV_COEF_I16) {
    const uint64_t warps = g.n_chunks < kMaxWarps ? g.n_chunks : kMaxWarps;
    w.n_slots = warps * kLanes * 2;   // two slot sets per warp: one coding, one awaiting placement
    w.slots_off = 0;
    w.state_off = align256(w.n_slots * g.slot_words * 2);
    w.ticket_off = w.state_off + align256(g.n_chunks * 8);
    w.total = w.ticket_off + 256;
    return w;
  }
  w.n_scan_blocks = (g.n_lanes + kScanPerBlock - 1) / kScanPerBlock;
  w.n_slots = g.n_lanes;
  w.slots_off = 0;
  w.lw_off = align256(g.n_lanes * g.slot_words * 2);
  w.part_off = w.lw_off + align256(g.n_lanes * 4);
  w.total = w.part_off + align256((w.n_scan_blocks + 1) * 8);
  return w;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Ordinals of four FP8 (two BF16) patterns at once: non-negative b -> b | top,
// negative b -> ~b.  prmt with selector nibbles 8..15 replicates the sign bit
// of a byte over the target byte, giving the per-lane mask in one instruction;
// the inverse takes the sign from the complemented ordinal.
__device__ __forceinline__ uint32_t sign_bytes8(uint32_t w) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"(w));
  return m;
}
__device__ __forceinline__ uint32_t sign_halves16(uint32_t w) {
  uint32_t m;
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(w));
  return m;
}
__device__ __forceinline__ uint32_t ord8x4(uint32_t w) { return w ^ (sign_bytes8(w) | 0x80808080u); }
__device__ __forceinline__ uint32_t unord8x4(uint32_t u) { return u ^ (sign_bytes8(~u) | 0x80808080u); }
__device__ __forceinline__ uint32_t ord16x2(uint32_t w) { return w ^ (sign_halves16(w) | 0x80008000u); }
__device__ __forceinline__ uint32_t unord16x2(uint32_t u) { return u ^ (sign_halves16(~u) | 0x80008000u); }

// streaming (evict-first) 128-bit loads and stores of the caches
__device__ __forceinline__ uint4 ldg_stream(const void* ptr) { return __ldcs(reinterpret_cast<const uint4*>(ptr)); }
__device__ __forceinline__ void stg_stream(void* ptr, uint4 v) { __stcs(reinterpret_cast<uint4*>(ptr), v); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
  return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

// scale bin of q = floor(beta * 2^16): 0 below 1/8, last bin from 32 up,
// otherwise octave * sub + linear sub-bin below the leading one
__device__ __forceinline__ uint32_t bin_from_q(uint64_t q, uint32_t sub) {
  const uint32_t sb = sub == 8 ? 3 : 2;
  if (q < (1ull << 13)) return 0;
  if (q >= (1ull << 21)) return 8 * sub - 1;
  const uint32_t pw = 63 - __clzll((long long)q);
  return sub * (pw - 13) + (uint32_t)((q >> (pw - sb)) & (sub - 1));
}

// base bin of the exponent model: the same grid extended upward without a cap
// (0 below 1/8); a position with prediction exponent e uses table
// min(max(base - 4 e, 0), 31)
__device__ __forceinline__ uint32_t bin_ext(uint64_t q) {
  if (q < (1ull << 13)) return 0;
  const uint32_t pw = 63 - __clzll((long long)q);
  return 4 * (pw - 13) + (uint32_t)((q >> (pw - 2)) & 3u);
}
__device__ __forceinline__ uint32_t vmin_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Exponent model (FP8): table byte offsets of a group's 16 positions from the
// lane's base bins (bw, four words of bytes) and the group's raw prediction
// words, two positions at a time in 16-bit lanes:
// base - min(base, 4 e) = max(base - 4 e, 0), then min with 31.
__device__ __forceinline__ void model_exp_word(uint32_t b, uint32_t w, uint32_t stride, uint32_t* t4) {
  const uint32_t e_ev = (w >> 1) & 0x003C003Cu, e_od = (w >> 9) & 0x003C003Cu;   // 4 e of bytes 0|2, 1|3
  const uint32_t b_ev = b & 0x00FF00FFu, b_od = (b >> 8) & 0x00FF00FFu;
  const uint32_t i_ev = vmin_u16x2(b_ev - vmin_u16x2(b_ev, e_ev), 0x001F001Fu);
  const uint32_t i_od = vmin_u16x2(b_od - vmin_u16x2(b_od, e_od), 0x001F001Fu);
  t4[0] = (i_ev & 0xFFFFu) * stride;
  t4[1] = (i_od & 0xFFFFu) * stride;
  t4[2] = (i_ev >> 16) * stride;
  t4[3] = (i_od >> 16) * stride;
}
__device__ __forceinline__ void model_exp_tables(const uint32_t* bw, const uint4& praw, uint32_t stride,
                                                 uint32_t* tb) {
#pragma unroll
  for (int k = 0; k < 4; ++k) model_exp_word(bw[k], word_of(praw, k), stride, tb + 4 * k);
}

// ---- checked build -----------------------------------------------------------
// With -DSKV_CHECKED=1 every shared-memory access of the codec kernels is
// checked against the launch's dynamic shared size and its natural alignment,
// and the encoder's table, word-buffer and scratch-slot cursors, the decoder's
// output rows, the chunk copy into the stream and the coefficient kernels'
// table indices against their own regions.  A failed check counts itself,
// records the first failing site and skips the access (a read gives 0); it
// never traps.  skv_checked_failures reads and clears the record.
#ifndef SKV_CHECKED
#define SKV_CHECKED 0
#endif
#if SKV_CHECKED
__device__ unsigned int g_check_count;
__device__ unsigned int g_check_site;
__device__ __noinline__ void check_fail(uint32_t site) {
  atomicAdd(&g_check_count, 1u);
  atomicCAS(&g_check_site, 0u, site);
}
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
  uint32_t v;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
  return v;
}
__device__ __forceinline__ bool smem_ok(uint32_t a, uint32_t n, uint32_t site) {
  const bool ok = (uint64_t)a + n <= dyn_smem_bytes() && (a & (n - 1)) == 0;
  if (!ok) check_fail(site);
  return ok;
}
#define SKV_CHECK(cond, site)        \
  do {                               \
    if (!(cond)) check_fail(site);   \
  } while (0)
#define SKV_SMEM_OK(a, n, site) smem_ok(a, n, site)
#else
#define SKV_CHECK(cond, site) \
  do {                        \
  } while (0)
#define SKV_SMEM_OK(a, n, site) true
#endif
// check sites (the value recorded for the first failure)
enum : uint32_t {
  kSiteSmemLoad = 1, kSiteSmemStore = 2, kSiteEncEntry = 3, kSiteWordBuffer = 4, kSiteScratchSlot = 5,
  kSiteStreamCopy = 6, kSiteDecOut = 7, kSiteRing = 8, kSiteCoefTable = 9
};

// ---- shared-memory access by byte offset into the dynamic shared array -----
// Plain C++ accesses (not volatile asm) so that the compiler may predicate and
// schedule them like any other instruction.
extern __shared__ __align__(16) uint8_t g_smem[];
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t v) {
  if (SKV_SMEM_OK(a, 2, kSiteSmemStore)) *reinterpret_cast<uint16_t*>(g_smem + a) = (uint16_t)v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  return SKV_SMEM_OK(a, 2, kSiteSmemLoad) ? *reinterpret_cast<const uint16_t*>(g_smem + a) : 0u;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) { return SKV_SMEM_OK(a, 1, kSiteSmemLoad) ? g_smem[a] : 0u; }
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  return SKV_SMEM_OK(a, 4, kSiteSmemLoad) ? *reinterpret_cast<const uint32_t*>(g_smem + a) : 0u;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t a) {
  return SKV_SMEM_OK(a, 8, kSiteSmemLoad) ? *reinterpret_cast<const uint2*>(g_smem + a) : make_uint2(0, 0);
}
__device__ __forceinline__ uint4 lds_u128(uint32_t a) {
  return SKV_SMEM_OK(a, 16, kSiteSmemLoad) ? *reinterpret_cast<const uint4*>(g_smem + a) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void sts_u128(uint32_t a, uint4 v) {
  if (SKV_SMEM_OK(a, 16, kSiteSmemStore)) *reinterpret_cast<uint4*>(g_smem + a) = v;
}
__device__ __forceinline__ void stg_u128(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Encoder entry {m_lo, w}, w = fr << 20 | cum << 8 | 1 << 7 | s with
// s = ceil(log2 fr): the reciprocal m = 2^32 + m_lo always has its top bit at
// 2^32, so floor(x / fr) = (umulhi(x, m_lo) + x) >> s (one multiply-add and a
// shift; the sum stays below 2^32 for x < fr 2^20).
__device__ __forceinline__ uint32_t enc_quot(uint32_t x, uint32_t m_lo, uint32_t w) {
  return __funnelshift_r(__umulhi(x, m_lo) + x, 0u, w);   // shift amount = w & 31 = s
}

// Constants held in registers (they come from the kernel arguments), so that
// the multiply-adds written with them stay on the FMA pipe: with literals the
// compiler turns them into shifts and adds on the integer ALU pipe, which the
// encoder's main loop keeps the busiest.
struct PipeConsts {
  uint32_t k4096, minus1, k2p20, k8;
};

// one coding step; renormalisation words go to a downward-growing buffer
// addressed by rp (shared-window byte address)
__device__ __forceinline__ void enc_step_smem(uint32_t& x, uint32_t& rp, uint2 e) {
  if (x >= (e.y & 0xFFF00000u)) {
    rp -= 2;
    sts_u16(rp, x);
    x >>= 16;
  }
  const uint32_t q = enc_quot(x, e.x, e.y);
  x = x + q * (4096u - (e.y >> 20)) + ((e.y >> 8) & 0xFFFu);
}
// The same step with the threshold fr << 20 and the multiplier 4096 - fr
// formed on the FMA pipe (both come from the entry, read ahead of the step,
// so the longer latency stays off the state's dependency chain).
__device__ __forceinline__ void enc_step_smem_fma(uint32_t& x, uint32_t& rp, uint2 e, const PipeConsts& k) {
  const uint32_t fr = e.y >> 20;
  if (x >= fr * k.k2p20) {
    rp -= 2;
    sts_u16(rp, x);
    x >>= 16;
  }
  const uint32_t q = enc_quot(x, e.x, e.y);
  x = x + q * (fr * k.minus1 + k.k4096) + ((e.y >> 8) & 0xFFFu);
}
// raw byte v as a uniform step (fr 16, cum 16 v), taken only where do_it holds
__device__ __forceinline__ void enc_raw_smem_if(uint32_t& x, uint32_t& rp, uint32_t v, bool do_it) {
  const bool ren = do_it && x >= (1u << 24);
  if (ren) {
    rp -= 2;
    sts_u16(rp, x);
  }
  const uint32_t xr = ren ? x >> 16 : x;
  const uint32_t xn = ((xr >> 4) << 12) | (xr & 15u) | (v << 4);
  x = do_it ? xn : x;
}
// a raw byte as a uniform step, words written downward straight into global scratch (COEF path)
__device__ __forceinline__ void enc_raw_gmem(uint32_t& x, uint16_t*& wp, uint32_t v) {
  if (x >= (1u << 24)) {
    *--wp = (uint16_t)x;
    x >>= 16;
  }
  x = ((x >> 4) << 12) | (x & 15u) | (v << 4);
}

// Decoder lane reading its words straight from global memory (COEF path).
struct DecLane {
  const uint16_t* w;
  uint32_t n, p, nxt, x;
};
__device__ __forceinline__ void dec_renorm(DecLane& L) {
  if (L.x < kStateLow) {
    L.x = __byte_perm(L.x, L.nxt, 0x1054);   // (x << 16) | nxt (nxt < 2^16)
    ++L.p;
    L.nxt = L.p < L.n ? L.w[L.p] : 0u;
  }
}
__device__ __forceinline__ uint32_t dec_raw(DecLane& L) {
  const uint32_t slot = L.x & 4095u;
  L.x = 16u * (L.x >> 12) + (slot & 15u);
  dec_renorm(L);
  return slot >> 4;
}
__device__ __forceinline__ void dec_open(DecLane& L, const uint8_t* bs, uint64_t a, uint64_t b, bool ok,
                                         uint32_t* status) {
  if (!ok) {
    atomicOr(status, SKV_FLAG_CORRUPT);
    L.w = nullptr; L.n = 0; L.p = 2; L.nxt = 0; L.x = kStateLow;
    return;
  }
  L.w = reinterpret_cast<const uint16_t*>(bs + a);
  L.n = (uint32_t)((b - a) >> 1);
  L.x = ((uint32_t)L.w[0] << 16) | L.w[1];
  L.p = 2;
  L.nxt = L.p < L.n ? L.w[L.p] : 0u;
  if (L.x < kStateLow) atomicOr(status, SKV_FLAG_CORRUPT);
}
__device__ __forceinline__ void dec_close(const DecLane& L, uint32_t* status) {
  if (L.x != kStateLow || L.p != L.n) atomicOr(status, SKV_FLAG_CORRUPT);
}

// Decoder lane reading its words through a 64-byte shared-memory ring of
// aligned 16-byte stream blocks (block k lives in ring slot k mod 4), filled
// by asynchronous copies: a refill first waits for the copies issued at the
// previous refill, then issues the blocks that keep [p/16, p/16 + 4) resident.
// A lane consumes at most 32 stream bytes between refills, so it never reads
// the block issued at the latest refill before the next one.  Offsets are
// relative to base = the lane's first byte rounded down to 64.
struct RingLane {
  const uint8_t* base; // bitstream + (lane start & ~63)
  uint32_t ring;       // shared-window address of the ring (64-byte aligned)
  uint32_t p;          // next word to consume
  uint32_t end;        // one past the lane's last byte
  uint32_t rb;         // next block to move into the ring
  uint32_t last;       // last block holding lane bytes (rb > last: nothing left)
  uint32_t nxt, x;
};
__device__ __forceinline__ uint4 load_block(const RingLane& L, uint32_t k) {
  return k <= L.last ? ldg_stream(L.base + ((uint64_t)k << 4)) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// asynchronous 4- / 8-byte copies from global memory to the dynamic shared
// array at byte offset a (waited for by cp_async_wait_all)
__device__ __forceinline__ void cp_async_4(uint32_t a, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(g_smem + a)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t a, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((uint32_t)__cvta_generic_to_shared(g_smem + a)),
               "l"(src)
               : "memory");
}
// block rb -> ring slot rb mod 4 (zero bytes read past the lane's last block)
__device__ __forceinline__ void ring_step(RingLane& L) {
  const uint32_t saddr = (uint32_t)__cvta_generic_to_shared(g_smem + L.ring + (L.rb & 3u) * 16u);
  if (!SKV_SMEM_OK(L.ring + (L.rb & 3u) * 16u, 16, kSiteRing)) return;
  const bool valid = L.rb <= L.last;
  const uint8_t* src = L.base + (valid ? ((uint64_t)L.rb << 4) : 0);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(src), "r"(valid ? 16u : 0u)
               : "memory");
  ++L.rb;
}
// make blocks [p/16, p/16 + 4) resident: one straight-line step covers a lane
// that moved into a new block since the last refill; lanes that moved further
// (escape-heavy stretches) catch up in a warp-uniform loop and wait for their
// copies at once
__device__ __forceinline__ void ring_refill(RingLane& L, uint32_t act) {
  cp_async_wait_all();
  uint32_t n = 0;
  if (L.rb < (L.p >> 4) + 4) { ring_step(L); ++n; }
  while (__any_sync(act, L.rb < (L.p >> 4) + 4)) {
    if (L.rb < (L.p >> 4) + 4) { ring_step(L); ++n; }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  if (n > 1) cp_async_wait_all();
}
__device__ __forceinline__ uint32_t ring_word(const RingLane& L, uint32_t p) {
  return lds_u16((p & (kRingBytes - 1)) + L.ring);
}
__device__ __forceinline__ void ring_renorm(RingLane& L) {
  if (L.x < kStateLow) {
    L.x = __byte_perm(L.x, L.nxt, 0x1054);   // (x << 16) | nxt in one PRMT (nxt < 2^16)
    L.p += 2;
    L.nxt = ring_word(L, L.p);
  }
}
// a raw byte (uniform step, fr 16) taken only where do_it holds
__device__ __forceinline__ uint32_t ring_raw_if(RingLane& L, bool do_it) {
  const uint32_t slot = L.x & 4095u;
  const uint32_t xn = 16u * (L.x >> 12) + (slot & 15u);
  const bool ren = do_it && xn < kStateLow;
  const uint32_t pn = L.p + 2;
  L.x = do_it ? (ren ? __byte_perm(xn, L.nxt, 0x1054) : xn) : L.x;
  if (ren) {
    L.p = pn;
    L.nxt = ring_word(L, pn);
  }
  return slot >> 4;
}
__device__ __forceinline__ void ring_open(RingLane& L, const uint8_t* bs, uint32_t ring, uint64_t a, uint64_t b,
                                          bool ok, uint32_t* status) {
  L.ring = ring;
  if (!ok) {   // nothing is read from global memory for a lane with bad offsets
    if (status) atomicOr(status, SKV_FLAG_CORRUPT);   // NULL: an idle lane, not an error
    L.base = bs;
    L.p = 0; L.end = 0; L.rb = 1; L.last = 0;
    L.x = kStateLow;
    L.nxt = 0;
    return;
  }
  const uint64_t a0 = a & ~63ull;
  L.base = bs + a0;
  L.p = (uint32_t)(a - a0);
  L.end = (uint32_t)(b - a0);
  L.last = (L.end - 1) >> 4;
  const uint32_t first = L.p >> 4;
  for (uint32_t k = first; k < first + 4; ++k)
    if (k <= L.last) sts_u128(ring + (k & 3u) * 16u, ldg_stream(L.base + ((uint64_t)k << 4)));
  L.rb = first + 4;
  L.x = (ring_word(L, L.p) << 16) | ring_word(L, L.p + 2);
  L.p += 4;
  L.nxt = ring_word(L, L.p);
  if (L.x < kStateLow && status) atomicOr(status, SKV_FLAG_CORRUPT);
}
// Reposition the ring at stream offset p (relative to base, at or after the
// lane's first byte): reload the four blocks from p's block on.
__device__ __forceinline__ void ring_reopen(RingLane& L, uint32_t p) {
  cp_async_wait_all();   // no earlier copy may still land in the ring
  const uint32_t first = p >> 4;
  for (uint32_t k = first; k < first + 4; ++k) sts_u128(L.ring + (k & 3u) * 16u, load_block(L, k));
  L.p = p;
  L.rb = first + 4;
}
__device__ __forceinline__ void ring_close(const RingLane& L, uint32_t* status) {
  if (L.x != kStateLow || L.p != L.end) atomicOr(status, SKV_FLAG_CORRUPT);
}

// Paged KV pools: pool (layer, k/v) holds n_blocks blocks of 2^shift tokens,
// each block [tokens][H][D]; bt[j] is the block of tokens [j 2^shift, (j+1) 2^shift).
// bt == nullptr means the dense [layer][k/v][head][token][D] layout.
struct Paged {
  const uint32_t* bt;
  uint32_t n_blocks, shift, H;
};
// Element index, in the paged pools, of token t, channel d of slice
// (layer, k/v, head); an out-of-range block-table entry flags SKV_FLAG_BAD_BLOCK
// and yields ok = false (the index then points into block 0).
__device__ __forceinline__ uint64_t paged_elem(const Paged& pg, uint64_t slice, uint64_t t, uint32_t d, uint32_t D,
                                               uint32_t* status, bool& ok) {
  const uint64_t lk = slice / pg.H, h = slice - lk * pg.H;
  uint32_t blk = __ldg(pg.bt + (t >> pg.shift));
  ok = blk < pg.n_blocks;
  if (!ok) {
    atomicOr(status, SKV_FLAG_BAD_BLOCK);
    blk = 0;
  }
  const uint64_t phys = ((uint64_t)blk << pg.shift) | (t & ((1ull << pg.shift) - 1));
  return (((lk * pg.n_blocks) << pg.shift) + phys) * ((uint64_t)pg.H * D) + h * D + d;
}

// The same from a block-table entry read earlier (the codec kernels read the
// entries of a lane's groups ahead of the group loads): lkb = (layer, k/v)
// pool's first row, hd0 = h * D + d0.
__device__ __forceinline__ uint64_t paged_elem_at(const Paged& pg, uint32_t blk, uint64_t t, uint64_t lkb,
                                                  uint64_t hd0, uint32_t D, uint32_t* status, bool& ok) {
  ok = blk < pg.n_blocks;
  if (!ok) {
    atomicOr(status, SKV_FLAG_BAD_BLOCK);
    blk = 0;
  }
  const uint64_t phys = ((uint64_t)blk << pg.shift) | (t & ((1ull << pg.shift) - 1));
  return (lkb + phys) * ((uint64_t)pg.H * D) + hd0;
}
__device__ __forceinline__ uint32_t paged_entry(const Paged& pg, uint64_t t) { return __ldg(pg.bt + (t >> pg.shift)); }

// lane offsets [a, b) of lane g, checked against the stream
__device__ __forceinline__ bool lane_span(const uint64_t* offs, uint64_t g, uint64_t n_lanes,
                                          uint64_t n_bytes, uint64_t* a, uint64_t* b) {
  *a = offs[g];
  *b = offs[g + 1];
  bool ok = *a <= *b && *b <= n_bytes && ((*a | *b) & 1) == 0 && *b - *a >= 4;
  if (g == 0 && *a != 0) ok = false;
  if (g + 1 == n_lanes && *b != n_bytes) ok = false;
  return ok;
}

// ---------------------------------------------------------------------------
// Table builder ([DCKV] how it differs: per-component Laplace integrated over
// the quantisation cells).  All integer, reproducible on any machine.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_build_tables(uint8_t* blob, uint32_t sub, int coef) {
  const uint32_t t = blockIdx.x, i = threadIdx.x;
  const uint32_t bin = coef ? t / 16 : t, f = coef ? t % 16 : 0;
  __shared__ unsigned long long P[kChain];
  __shared__ uint32_t rem[256];
  __shared__ uint32_t cums[257];
  __shared__ uint32_t red[8];
  if (i == 0) {
    // representative scale: midpoint of the sub-bin, Q16
    const uint32_t e = bin / sub, j = bin % sub;
    const uint64_t bq = ((1ull << (e + 13)) / (2ull * sub)) * (2ull * sub + 2ull * j + 1ull);
    const uint64_t xq = ((1ull << 44) + (bq >> 1)) / bq;  // Q32 of 1/(16 beta)
    uint64_t a = 1ull << 32;
    long long tau = (long long)a;
    for (uint64_t n = 1; n <= 15; ++n) {                  // exp(-x) by Taylor
      a = (a * xq + n * (1ull << 31)) / (n << 32);
      tau += (n & 1) ? -(long long)a : (long long)a;
    }
    const uint64_t tq = (uint64_t)tau;
    P[0] = 1ull << 32;
    for (uint32_t n = 1; n < kChain; ++n) P[n] = (P[n - 1] * tq + (1ull << 31)) >> 32;
  }
  __syncthreads();
  auto F = [&](long long n) -> uint64_t {   // Laplace CDF at n/16 from the mean, Q32
    return n < 0 ? (P[-n] >> 1) : ((1ull << 32) - (P[n] >> 1));
  };
  uint64_t m;
  if (i < 255) {
    const long long s = (long long)i - 127;
    m = F(16 * s + 8 - (long long)f) - F(16 * s - 8 - (long long)f);
  } else {
    m = F(-16 * 127 - 8 - (long long)f) + ((1ull << 32) - F(16 * 127 + 8 - (long long)f));
  }
  const uint64_t scaled = m * 3840ull;
  uint32_t fr = 1u + (uint32_t)(scaled >> 32);
  const uint32_t rm = (uint32_t)scaled;
  rem[i] = rm;
  // block sum of the floors
  uint32_t s = fr;
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if ((i & 31) == 0) red[i >> 5] = s;
  __syncthreads();
  uint32_t total = 0;
  for (int k = 0; k < 8; ++k) total += red[k];
  const uint32_t deficit = 4096u - total;
  // largest remainders get one more unit; ties go to the lower symbol
  uint32_t rank = 0;
  for (uint32_t k = 0; k < 256; ++k) {
    const uint32_t r2 = rem[k];
    rank += (r2 > rm) || (r2 == rm && k < i);
  }
  fr += rank < deficit ? 1u : 0u;
  // exclusive scan of fr
  uint32_t incl = fr;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if ((i & 31) >= (uint32_t)o) incl += v;
  }
  __syncthreads();
  if ((i & 31) == 31) red[i >> 5] = incl;
  __syncthreads();
  uint32_t base = 0;
  for (uint32_t k = 0; k < (i >> 5); ++k) base += red[k];
  const uint32_t cum = base + incl - fr;
  cums[i] = cum;
  if (i == 255) cums[256] = 4096;
  uint8_t* tb = blob + (uint64_t)t * SKV_TABLE_STRIDE;
  reinterpret_cast<uint16_t*>(tb + SKV_TABLE_FREQ_OFF)[i] = (uint16_t)fr;
  reinterpret_cast<uint16_t*>(tb + SKV_TABLE_CUM_OFF)[i] = (uint16_t)cum;
  if (i == 255) reinterpret_cast<uint16_t*>(tb + SKV_TABLE_CUM_OFF)[256] = 4096;
  // encoder reciprocal: s = ceil(log2 fr), m = ceil(2^(32+s)/fr) in [2^32, 2^33).
  // floor(x m / 2^(32+s)) = floor(x / fr) for all x < fr 2^20, since the error
  // term (fr 2^20 - 1)(m fr - 2^(32+s)) < fr^2 2^20 <= 2^(32+s) for s <= 12,
  // and x m < 2^64 there
  uint32_t sh = 0;
  while ((1u << sh) < fr) ++sh;
  const uint64_t mm = ((1ull << (32 + sh)) + fr - 1) / fr;
  uint2 enc;
  enc.x = (uint32_t)mm;
  enc.y = (fr << 20) | (cum << 8) | (1u << 7) | sh;
  reinterpret_cast<uint2*>(tb + SKV_TABLE_ENC_OFF)[i] = enc;
  // decoder entry: fr, and -cum as a signed upper half (the update adds it)
  reinterpret_cast<uint32_t*>(tb + SKV_TABLE_DEC_OFF)[i] = fr | ((0u - cum) << 16);
  __syncthreads();
  // slot -> symbol: the last symbol whose cum <= slot
  uint8_t* lut = tb + SKV_TABLE_LUT_OFF;
  for (uint32_t k = 0; k < 16; ++k) {
    const uint32_t slot = i * 16 + k;
    uint32_t lo = 0, hi = 256;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (cums[mid] <= slot) lo = mid; else hi = mid;
    }
    lut[slot] = (uint8_t)lo;
    if (coef)
      reinterpret_cast<uint32_t*>(blob + (uint64_t)gridDim.x * SKV_TABLE_STRIDE + (uint64_t)t * SKV_TABLE_SLOT_BYTES)[slot] =
          lo | ((cums[lo + 1] - cums[lo]) << 8) | ((slot - cums[lo]) << 20);
  }
}

// ---------------------------------------------------------------------------
// Calibration ([SKV] which predictor: statistics measured once on calibration
// tokens and frozen).  One CTA per slice, each thread covers 16-byte groups of
// channels for a stride of tokens; partial sums are combined across the lanes
// that share a channel group with warp shuffles, then across warps.
// ---------------------------------------------------------------------------
template <int ESZ, bool PAGED>
__global__ void __launch_bounds__(256) k_calibrate_kv(const uint8_t* tgt, const uint8_t* prd,
                                                      uint8_t* bins, uint32_t* sum_abs,
                                                      uint32_t* hist, uint64_t T, uint32_t D,
                                                      uint32_t nc, Paged pg, uint32_t* status, uint32_t model) {
  constexpr int G = 16 / ESZ;
  __shared__ unsigned long long S[512];
  const uint64_t slice = blockIdx.x;
  const uint32_t nv = D / G;                    // 16-byte groups per token (<= 32)
  const uint32_t tid = threadIdx.x;
  const uint32_t cg = tid % nv, tph = tid / nv, nph = blockDim.x / nv;
  for (uint32_t d = tid; d < D; d += blockDim.x) S[d] = 0;
  __syncthreads();
  unsigned long long acc[G];   // model 1 adds |r| 2^e: up to 2^23 per token
#pragma unroll
  for (int e = 0; e < G; ++e) acc[e] = 0;
  const uint64_t base = slice * T * D;          // element index of the slice
  if (tph < nph) {
    for (uint64_t t = tph; t < nc; t += nph) {
      bool ok = true;
      const uint64_t el = PAGED ? paged_elem(pg, slice, t, cg * G, D, status, ok) : base + t * D + (uint64_t)cg * G;
      const uint4 tv = ldg_stream(tgt + el * ESZ), pv = ldg_stream(prd + el * ESZ);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t a = ESZ == 1 ? ord8x4(word_of(tv, k)) : ord16x2(word_of(tv, k));
        const uint32_t b = ESZ == 1 ? ord8x4(word_of(pv, k)) : ord16x2(word_of(pv, k));
#pragma unroll
        for (int h = 0; h < 4 / ESZ; ++h) {
          const uint32_t sh = 8 * ESZ * h, mk = ESZ == 1 ? 0xFFu : 0xFFFFu;
          const int r = (int)((a >> sh) & mk) - (int)((b >> sh) & mk);
          const int e = k * (4 / ESZ) + h;
          const uint32_t ex = model ? (word_of(pv, k) >> (sh + 3)) & 15u : 0u;   // prediction's exponent field
          acc[e] += (unsigned long long)(uint32_t)(r < 0 ? -r : r) << ex;
          if (hist) {
            const uint32_t sym = (r >= -127 && r <= 127) ? (uint32_t)(r + 127) : 255u;
            atomicAdd(&hist[((slice * D) + (uint64_t)cg * G + e) * 256 + sym], 1u);
          }
        }
      }
    }
  }
  // lanes tid, tid + nv, ... of one warp share a channel group
#pragma unroll
  for (int e = 0; e < G; ++e) {
    unsigned long long v = acc[e];
    for (uint32_t o = nv; o < 32; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    acc[e] = v;
  }
  if ((tid & 31) < nv && tph < nph) {
#pragma unroll
    for (int e = 0; e < G; ++e) atomicAdd(&S[cg * G + e], acc[e]);
  }
  __syncthreads();
  for (uint32_t d = tid; d < D; d += blockDim.x) {
    const uint64_t sv = S[d];
    const uint64_t q = nc ? (sv << 16) / nc : 0;
    bins[slice * D + d] = (uint8_t)(model ? bin_ext(q) : bin_from_q(q, 4));
    if (sum_abs) sum_abs[slice * D + d] = sv > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)sv;
  }
}

// COEF: bins from beta = scale/step; below 0.05 the component is switched off
// ([DCKV] how it works)
__global__ void k_calibrate_coef(const float* beta, uint8_t* bins, uint32_t C) {
  const uint32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  const float b = beta[c];
  uint8_t out;
  if (!(b >= 0.05f)) out = 0xFF;
  else if (b >= 32.0f) out = 63;
  else out = (uint8_t)bin_from_q((uint64_t)floorf(__fmul_rn(b, 65536.0f)), 8);
  bins[c] = out;
}

// ---------------------------------------------------------------------------
// Encoder, KV caches.  Persistent warps take chunks from an atomic ticket.
// Lane l of a chunk owns 16-byte groups l, l + 32, ...; the reverse pass walks
// them from the last group down, prefetching the next group's 128-bit loads.
// ---------------------------------------------------------------------------
struct CodecArgs {
  const uint8_t* tgt;   // encode: target; decode: unused
  const uint8_t* prd;   // prediction (COEF: mu)
  uint8_t* out;         // decode: target output
  const uint8_t* tables;
  const uint8_t* bins;
  uint16_t* slots;      // encode scratch
  uint32_t* lane_words;
  const uint8_t* bs;    // decode: bitstream
  const uint64_t* offs; // decode: lane offsets
  uint64_t n_bytes;
  uint32_t* status;
  uint64_t n_chunks, cps, slice_pos, n_lanes, slot_words;
  uint32_t K, D, C;
  // encode, KV: fused look-back placement
  unsigned long long* chunk_state;  // per chunk: flag << 62 | bytes
  unsigned long long* ticket;       // next chunk to hand out
  uint64_t* lane_offsets;
  uint8_t* out_bs;                  // final bitstream
  uint64_t cap;
  uint64_t slot_warps;              // warps that own a slot set in the workspace
  uint64_t last_wave;               // chunks from here on are the last wave handed out
  Paged pg;                         // paged pools (pg.bt == nullptr: dense caches)
  PipeConsts k;                     // 4096, 0xFFFFFFFF, 2^20, 8 (see PipeConsts)
};

template <int ESZ>
__device__ __forceinline__ void load_lane_tables(const CodecArgs& a, uint64_t slice, uint32_t d0,
                                                 uint32_t stride, uint32_t* tb) {
  constexpr int G = 16 / ESZ;
  const uint8_t* bp = a.bins + slice * a.D + d0;
  uint32_t bw[4];
  if (G == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(bp);
    bw[0] = v.x; bw[1] = v.y; bw[2] = v.z; bw[3] = v.w;
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(bp);
    bw[0] = v.x; bw[1] = v.y; bw[2] = 0; bw[3] = 0;
  }
  bool bad = false;
#pragma unroll
  for (int e = 0; e < G; ++e) {
    uint32_t b = (bw[e >> 2] >> (8 * (e & 3))) & 0xFFu;
    if (b >= kKvTables) { bad = true; b = kKvTables - 1; }
    tb[e] = b * stride;
  }
  if (bad) atomicOr(a.status, SKV_FLAG_BAD_BIN);
}

// exponent model: the lane's 16 base bins as four words of bytes
__device__ __forceinline__ void load_lane_bases(const CodecArgs& a, uint64_t slice, uint32_t d0, uint32_t* bw) {
  const uint4 v = *reinterpret_cast<const uint4*>(a.bins + slice * a.D + d0);
  bw[0] = v.x; bw[1] = v.y; bw[2] = v.z; bw[3] = v.w;
}

// Flush the oldest complete 16-byte blocks of every lane's word buffer (the
// top of the downward-growing buffer) to the lane's global scratch slot,
// downward from gp; the remaining partial block moves to the top.  All lanes
// in act call it together, so the warp pays for one flush loop at a time.
__device__ __forceinline__ void emit_flush_sync(uint32_t act, uint32_t buf_top, uint32_t& rp, uint8_t*& gp) {
  const uint32_t fill = buf_top - rp;
  const uint32_t nb = fill >> 4, rem = fill & 15u;
  const uint32_t nmax = __reduce_max_sync(act, nb);
  for (uint32_t j = 1; j <= nmax; ++j)
    if (j <= nb) stg_u128(gp - 16 * j, lds_u128(buf_top - 16 * j));
  gp -= 16 * nb;
  if (nb != 0 && rem != 0) sts_u128(buf_top - 16, lds_u128(buf_top - 16 * nb - 16));
  rp = buf_top - rem;
}
// Final flush of one lane: every block, the lowest one padded below the
// lane's first word.
__device__ __forceinline__ void emit_flush_all(uint32_t buf_top, uint32_t rp, uint8_t*& gp) {
  const uint32_t nb = (buf_top - rp + 15) >> 4;
  for (uint32_t j = 1; j <= nb; ++j) stg_u128(gp - 16 * j, lds_u128(buf_top - 16 * j));
  gp -= 16 * nb;
}

// max of the unsigned 16-bit halves
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---- mbarriers (shared memory, one arrival + transaction bytes) ----------
constexpr uint64_t kBarWaitNs = 1000000000ull;   // ~1 s bound on every barrier wait
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// wait for the phase of parity `parity` to complete; false after ~1 s
__device__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try(bar, parity))
    if (global_ns() - t0 > kBarWaitNs) return false;
  return true;
}
// bulk copy of `bytes` (a multiple of 16) from global src to shared dst, both
// 16-byte aligned, completing its bytes on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---- decoupled look-back over chunks -------------------------------------
// chunk_state[c] = flag << 62 | value: flag 1 = the chunk's byte total is
// published, 2 = the inclusive prefix (bytes of chunks 0..c) is published,
// 3 = a predecessor failed.  Chunks are handed out in increasing order by an
// atomic ticket, so every chunk a warp waits on is held by a running warp.
constexpr unsigned long long kStAgg = 1ull << 62, kStInc = 2ull << 62, kStErr = 3ull << 62;
constexpr unsigned long long kStVal = (1ull << 62) - 1;
constexpr uint32_t kMaxSpins = 1u << 21;   // ~1 s of polling before giving up

__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum64(unsigned long long v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Publish chunk c's byte total (whole warp calls): chunk 0 publishes its
// inclusive prefix at once, every other chunk its aggregate.
__device__ __forceinline__ void chunk_publish(unsigned long long* st, uint64_t c, unsigned long long total) {
  if ((threadIdx.x & 31) == 0) st_release(&st[c], (c == 0 ? kStInc : kStAgg) | total);
}

// Exclusive byte prefix of chunk c, whose aggregate is already published
// (whole warp calls): walks back over the predecessors 32 at a time, adding
// aggregates until an inclusive prefix, waiting (bounded) on any that is
// still coding; then publishes c's inclusive prefix.  ~0 if it failed.
// The batch where the walk stops also gets its walked chunks' inclusive
// prefixes published (each one is the found prefix plus the aggregates below
// it in the batch, the value any later walk would compute), so that walks
// from later chunks stop sooner.
__device__ unsigned long long chunk_resolve(unsigned long long* st, uint64_t c, unsigned long long total,
                                            uint32_t* status, uint32_t max_spins) {
  const uint32_t tid = threadIdx.x & 31;
  if (c == 0) return 0;
  unsigned long long excl = 0;
  long long j = (long long)c - 1;
  uint32_t spins = 0;
  bool failed = false;
  while (true) {
    const long long idx = j - (long long)tid;
    const unsigned long long v = idx >= 0 ? ld_acquire(&st[idx]) : kStInc;
    const uint32_t flag = (uint32_t)(v >> 62);
    const uint32_t stop = __ballot_sync(0xFFFFFFFFu, flag >= 2);   // inclusive or failed
    const uint32_t none = __ballot_sync(0xFFFFFFFFu, flag == 0);
    const uint32_t upto = stop ? ((2u << (__ffs(stop) - 1)) - 1) : 0xFFFFFFFFu;   // lanes 0..first stop
    if (none & upto) {                                              // a predecessor is still coding
      if (++spins > max_spins) { failed = true; break; }
      __nanosleep(100);
      continue;
    }
    if (stop && ((v >> 62) == 3) && tid == (uint32_t)(__ffs(stop) - 1)) failed = true;
    failed = __any_sync(0xFFFFFFFFu, failed);
    if (failed) break;
    const unsigned long long mine = ((upto >> tid) & 1) ? (v & kStVal) : 0ull;
    if (stop) {
      // suffix sums over lanes tid..first stop: the inclusive prefix of chunk j - tid
      unsigned long long suf = mine;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long u = __shfl_down_sync(0xFFFFFFFFu, suf, o);
        if (tid + o < 32) suf += u;
      }
      const uint32_t s0 = (uint32_t)(__ffs(stop) - 1);
      if (tid < s0 && idx >= 0) st_release(&st[idx], kStInc | suf);
      excl += __shfl_sync(0xFFFFFFFFu, suf, 0);
      break;
    }
    excl += warp_sum64(mine);
    j -= 32;
  }
  if (failed) {
    if (tid == 0) {
      atomicOr(status, SKV_FLAG_TIMEOUT);
      st_release(&st[c], kStErr);
    }
    return ~0ull;
  }
  if (tid == 0) st_release(&st[c], kStInc | (excl + total));
  return excl;
}

// Both steps at once (the self-test's use).
__device__ unsigned long long chunk_lookback(unsigned long long* st, uint64_t c, unsigned long long total,
                                             uint32_t* status, uint32_t max_spins) {
  chunk_publish(st, c, total);
  return chunk_resolve(st, c, total, status, max_spins);
}

// Warp-cooperative copy of n_w 16-bit words from src to dst (both 2-byte
// aligned): 32-bit accesses, a 16-bit funnel when the two differ by 2 mod 4,
// sixteen independent loads in flight per thread (the copy is latency bound);
// streaming loads and stores (neither side is read again by this kernel).
__device__ __forceinline__ void warp_copy_words(uint16_t* dst, const uint16_t* src, uint32_t n_w, uint32_t tid) {
  if (n_w == 0) return;
  if ((reinterpret_cast<uintptr_t>(dst) & 3) != 0) {   // make dst 4-byte aligned
    if (tid == 0) dst[0] = src[0];
    ++dst; ++src; --n_w;
  }
  const uint32_t n32 = n_w >> 1;
  uint32_t* d32 = reinterpret_cast<uint32_t*>(dst);
  if ((reinterpret_cast<uintptr_t>(src) & 3) == 0) {
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src);
    for (uint32_t k0 = 0; k0 < n32; k0 += 512) {
      uint32_t v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t k = k0 + u * 32 + tid;
        v[u] = k < n32 ? __ldcs(s32 + k) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t k = k0 + u * 32 + tid;
        if (k < n32) __stcs(d32 + k, v[u]);
      }
    }
  } else {
    const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src - 1);   // aligned, one word early
    for (uint32_t k0 = 0; k0 < n32; k0 += 512) {
      uint32_t lo[16], hi[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t k = k0 + u * 32 + tid;
        lo[u] = k < n32 ? __ldcs(s32 + k) : 0u;
        hi[u] = k < n32 ? __ldcs(s32 + k + 1) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t k = k0 + u * 32 + tid;
        if (k < n32) __stcs(d32 + k, __funnelshift_r(lo[u], hi[u], 16));
      }
    }
  }
  if ((n_w & 1) && tid == 0) dst[n_w - 1] = src[n_w - 1];
}

// A chunk's lanes are copied from their scratch slots into the stream in
// one of two ways.  While other chunks are still being coded, the copy above
// runs lane after lane: its memory latency is hidden by the SM's other warps
// and it costs no shared-memory cycles, which coding needs.  Placements made
// once the last chunks have been handed out have no such cover, so chunks of
// at most kStagedMaxBytes (a few staging rounds instead of 32 lane round
// trips) copy through staging slots (the warp's word buffers, idle between
// chunks); larger chunks measured faster with the lane-by-lane copy.  Each
// lane's source bytes, widened to whole 16-byte blocks (the slot ends on a
// block boundary), are cut into pieces of at most kCpPiece bytes; up to
// kCpSlots pieces are in flight at once as bulk copies, each completing on its
// own mbarrier, so the chunk costs a few memory round trips instead of one
// per lane.  A landed piece is written out as aligned 16-byte destination
// blocks, each assembled from two 16-byte shared-memory reads shifted by the
// piece's (even) byte offset; the 16-bit words at either end that share a
// destination block with another piece, lane or chunk are written one by one.
constexpr uint32_t kCpSlots = 4, kCpPiece = 1024, kCpStride = 1152;
constexpr uint32_t kStagedMaxBytes = 32768;
static_assert(kCpSlots * kCpStride <= kLanes * kEmitBytes, "staging slots fit in a warp's word buffers");
static_assert(kCpStride >= kCpPiece + 16 && kCpStride % 16 == 0, "the shifted block reads end 16 bytes past a piece");
static_assert(kCpSlots <= 32, "one descriptor-holding thread per slot");
constexpr uint32_t kEncWarpExtra = kCpSlots * 8;   // a warp's staging mbarriers, after all the word buffers
// shared-memory byte offsets of warp w's staging slots (its word buffers) and mbarriers
__device__ __forceinline__ uint32_t enc_stage_at(uint32_t w) { return kEncTabBytes + w * (kLanes * kEmitBytes); }
__device__ __forceinline__ uint32_t enc_bars_at(uint32_t w, uint32_t threads) {
  return kEncTabBytes + threads * kEmitBytes + w * kEncWarpExtra;
}
__host__ __device__ constexpr uint32_t enc_smem_bytes(uint32_t threads) {
  return kEncTabBytes + threads * kEmitBytes + threads / 32 * kEncWarpExtra;
}
static_assert(enc_smem_bytes(kEncThreads) <= 227 * 1024, "the encoder's shared memory fits one CTA per SM");
constexpr uint32_t kPlaceFailed = 1u << 31;       // place_chunk: a staging wait gave up

// 16 destination bytes from the 32 staged bytes w[0..7] starting at byte
// 4 q + 2 h (q, h warp-uniform)
__device__ __forceinline__ uint4 shift_block(const uint4& lo, const uint4& hi, uint32_t q, uint32_t h) {
  const uint32_t sh = h ? 16u : 0u;
  uint32_t v0, v1, v2, v3, v4;
  if (q == 0) { v0 = lo.x; v1 = lo.y; v2 = lo.z; v3 = lo.w; v4 = hi.x; }
  else if (q == 1) { v0 = lo.y; v1 = lo.z; v2 = lo.w; v3 = hi.x; v4 = hi.y; }
  else if (q == 2) { v0 = lo.z; v1 = lo.w; v2 = hi.x; v3 = hi.y; v4 = hi.z; }
  else { v0 = lo.w; v1 = hi.x; v2 = hi.y; v3 = hi.z; v4 = hi.w; }
  return make_uint4(__funnelshift_r(v0, v1, sh), __funnelshift_r(v1, v2, sh), __funnelshift_r(v2, v3, sh),
                    __funnelshift_r(v3, v4, sh));
}

// Resolve a coded chunk's byte offset (its total is published) and write its
// lane offsets (whole warp calls).  Returns this thread's format lane's
// stream offset, or ~0 when the chunk is not to be copied (a failed wait or
// a stream past the capacity, both flagged).
__device__ __forceinline__ unsigned long long chunk_lane_offset(const CodecArgs& a, unsigned long long chunk,
                                                                unsigned long long total, uint32_t len,
                                                                uint32_t incl) {
  const uint32_t tid = threadIdx.x & 31;
  const unsigned long long excl = chunk_resolve(a.chunk_state, chunk, total, a.status, kMaxSpins);
  if (excl == ~0ull) return ~0ull;
  const unsigned long long lane_off = excl + incl - len;
  a.lane_offsets[chunk * kLanes + tid] = lane_off;
  if (chunk + 1 == a.n_chunks && tid == 31) a.lane_offsets[a.n_lanes] = excl + total;
  if (excl + total > a.cap) {
    if (tid == 0) atomicOr(a.status, SKV_FLAG_CAPACITY);
    return ~0ull;
  }
  return lane_off;
}

// Place a coded chunk whose total is published (whole warp calls): resolve
// its byte offset, write its lane offsets, copy its 32 lane streams from the
// slot set `sset` into the bitstream lane after lane.  len / incl are this
// thread's format lane length and inclusive prefix within the chunk.
__device__ __forceinline__ void place_chunk(const CodecArgs& a, unsigned long long chunk, unsigned long long total,
                                            uint32_t len, uint32_t incl, uint64_t sset, uint32_t CS, uint32_t R) {
  const uint32_t tid = threadIdx.x & 31;
  const unsigned long long lane_off = chunk_lane_offset(a, chunk, total, len, incl);
  if (lane_off == ~0ull) return;
  __syncwarp();
  for (uint32_t l = 0; l < kLanes; ++l) {
    const uint32_t n_w = __shfl_sync(0xFFFFFFFFu, len, l) >> 1;
    const unsigned long long dst = __shfl_sync(0xFFFFFFFFu, lane_off, l);
    const uint32_t owner = (l % CS) * R + l / CS;
    SKV_CHECK(dst + 2ull * n_w <= a.cap && 2ull * n_w <= 2 * a.slot_words, kSiteStreamCopy);
    const uint16_t* src = reinterpret_cast<const uint16_t*>(
        reinterpret_cast<const uint8_t*>(a.slots + (sset * kLanes + owner + 1) * a.slot_words)) - n_w;
    warp_copy_words(reinterpret_cast<uint16_t*>(a.out_bs + dst), src, n_w, tid);
  }
  __syncwarp();
}

// The same through the staging slots.  phase: the next parities of the
// warp's staging mbarriers, returned updated, with kPlaceFailed set if a wait
// gave up (status flagged, every copy waited for).
__device__ __forceinline__ uint32_t place_chunk_staged(const CodecArgs& a, unsigned long long chunk,
                                                       unsigned long long total, uint32_t len, uint32_t incl,
                                                       uint64_t sset, uint32_t CS, uint32_t R, uint32_t phase) {
  const uint32_t tid = threadIdx.x & 31;
  const unsigned long long lane_off = chunk_lane_offset(a, chunk, total, len, incl);
  if (lane_off == ~0ull) return phase;
  const uint32_t owner = (tid % CS) * R + tid / CS;
  const uint8_t* end = reinterpret_cast<const uint8_t*>(a.slots + (sset * kLanes + owner + 1) * a.slot_words);
  SKV_CHECK(lane_off + len <= a.cap && len <= 2 * a.slot_words, kSiteStreamCopy);
  const uint32_t span = min((len + 15u) & ~15u, (uint32_t)(2 * a.slot_words));   // aligned source bytes
  const uint32_t np = (span + kCpPiece - 1) / kCpPiece;
  uint32_t pincl = np;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, pincl, o);
    if (tid >= (uint32_t)o) pincl += u;
  }
  const uint32_t n_pieces = __shfl_sync(0xFFFFFFFFu, pincl, 31);
  const uint32_t sbase = smem_addr(g_smem);
  const uint32_t stage = enc_stage_at(threadIdx.x >> 5), bars = enc_bars_at(threadIdx.x >> 5, blockDim.x);
  // the slots were written, and the staging area (the word buffers) last
  // read, by this warp's ordinary accesses; the bulk copies go through the
  // asynchronous proxy
  asm volatile("fence.proxy.async;" ::: "memory");
  __syncwarp();
  // thread s keeps the write-out of the piece in slot s: destination start
  // (an address: the stream itself need only be 2-byte aligned), staged
  // offset of its first byte, byte count
  unsigned long long my_d0 = 0;
  uint32_t my_s0 = 0, my_n = 0;
  uint32_t q_in = 0;
  auto slot_at = [&](uint32_t slot) -> uint32_t { return stage + slot * kCpStride; };
  auto issue = [&]() {
    // piece q_in: its lane is the number of lanes whose inclusive piece count is at most q_in
    const uint32_t l = __popc(__ballot_sync(0xFFFFFFFFu, pincl <= q_in)) & 31u;
    const uint32_t k = q_in - __shfl_sync(0xFFFFFFFFu, pincl - np, l);
    const uint32_t sp = __shfl_sync(0xFFFFFFFFu, span, l);
    const uint32_t len_l = __shfl_sync(0xFFFFFFFFu, len, l);
    const unsigned long long dst_l = __shfl_sync(0xFFFFFFFFu, lane_off, l);
    const uint8_t* end_l = reinterpret_cast<const uint8_t*>(
        __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(end), l));
    const uint32_t lo = k * kCpPiece, bytes = min(kCpPiece, sp - lo);   // source bytes [lo, lo + bytes) of the span
    const uint32_t pad = sp - len_l;                                    // span bytes before the lane's first byte
    const uint32_t v0 = lo > pad ? lo : pad;                            // first lane byte in the piece
    const uint32_t slot = q_in % kCpSlots;
    const uint8_t* src = end_l - sp + lo;
    const uint32_t sa = slot_at(slot);
    SKV_CHECK(SKV_SMEM_OK(sa, 16, kSiteStreamCopy) && SKV_SMEM_OK(sa + kCpStride - 16, 16, kSiteStreamCopy) &&
                  bytes % 16 == 0 &&
                  bytes <= kCpPiece && pad < 16 && sp <= 2 * a.slot_words,
              kSiteStreamCopy);
    if (tid == slot) {
      my_d0 = reinterpret_cast<unsigned long long>(a.out_bs) + dst_l + (v0 - pad);
      my_s0 = sa + (v0 - lo);
      my_n = lo + bytes - v0;
    }
    if (tid == 0) {
      mbar_expect_tx(sbase + bars + 8 * slot, bytes);
      bulk_g2s(sbase + sa, src, bytes, sbase + bars + 8 * slot);
    }
    ++q_in;
  };
  while (q_in < n_pieces && q_in < kCpSlots) issue();
  uint32_t q = 0;
  for (; q < n_pieces; ++q) {
    const uint32_t slot = q % kCpSlots;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(sbase + bars + 8 * slot, (phase >> slot) & 1u))) break;
    phase ^= 1u << slot;
    const unsigned long long d0 = __shfl_sync(0xFFFFFFFFu, my_d0, slot);
    const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, my_s0, slot);
    const uint32_t n = __shfl_sync(0xFFFFFFFFu, my_n, slot);
    const unsigned long long d1 = d0 + n;
    const unsigned long long da = (d0 + 15) & ~15ull, db = d1 & ~15ull;
    if (da < db) {
      // whole destination blocks [da, db), staged from s0 + (da - d0)
      const uint32_t sa = s0 + (uint32_t)(da - d0);
      const uint32_t base = sa & ~15u, q4 = (sa >> 2) & 3u, h = (sa >> 1) & 1u;
      const uint32_t nb = (uint32_t)((db - da) >> 4);
      uint4* dst = reinterpret_cast<uint4*>(da);
      for (uint32_t i = tid; i < nb; i += 32) {
        const uint4 lo4 = lds_u128(base + 16 * i), hi4 = lds_u128(base + 16 * i + 16);
        __stcs(dst + i, shift_block(lo4, hi4, q4, h));
      }
      // the 16-bit words before da and from db on
      const uint32_t nh = (uint32_t)(da - d0) >> 1, nt = (uint32_t)(d1 - db) >> 1;
      if (tid < nh) *reinterpret_cast<uint16_t*>(d0 + 2 * tid) = (uint16_t)lds_u16(s0 + 2 * tid);
      else if (tid >= 8 && tid - 8 < nt)
        *reinterpret_cast<uint16_t*>(db + 2 * (tid - 8)) = (uint16_t)lds_u16(s0 + (uint32_t)(db - d0) + 2 * (tid - 8));
    } else {
      // fewer than two blocks' worth: 16-bit words only
      for (uint32_t i = tid; i < (n >> 1); i += 32)
        *reinterpret_cast<uint16_t*>(d0 + 2 * i) = (uint16_t)lds_u16(s0 + 2 * i);
    }
    // every read of the slot is done before the next bulk copy overwrites it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (q_in < n_pieces) issue();
  }
  if (q < n_pieces) {
    // a wait gave up: flag it, then wait (bounded) for the copies still in flight
    if (tid == 0) atomicOr(a.status, SKV_FLAG_TIMEOUT);
    for (; q < q_in; ++q) {
      const uint32_t slot = q % kCpSlots;
      __all_sync(0xFFFFFFFFu, mbar_wait(sbase + bars + 8 * slot, (phase >> slot) & 1u));
      phase ^= 1u << slot;
    }
    return phase | kPlaceFailed;
  }
  return phase;
}

// Place the warp's pending chunk (whole warp calls): through the staging
// slots when no later chunk is left to hand out (last) and the chunk is
// small enough, lane after lane otherwise.  Returns the staging mbarriers'
// parities (see place_chunk_staged).
__device__ __noinline__ uint32_t place_pending(const CodecArgs& a, unsigned long long chunk, unsigned long long total,
                                               uint32_t len, uint32_t incl, uint64_t sset, uint32_t CS, uint32_t R,
                                               bool last, uint32_t phase) {
  if (last && total <= kStagedMaxBytes) return place_chunk_staged(a, chunk, total, len, incl, sset, CS, R, phase);
  place_chunk(a, chunk, total, len, incl, sset, CS, R);
  return phase;
}

template <int ESZ, bool PAGED, bool MODEL>
__global__ void __launch_bounds__(kEncThreads, 1) k_encode_kv(CodecArgs a) {
  constexpr int G = 16 / ESZ;
  // Room the word buffer must have before a group: a symbol step emits at
  // most one word, an escaped position adds at most ESZ raw words.
  constexpr uint32_t kRoomPlain = kEmitBytes - 2 * G;
  constexpr uint32_t kRoomEsc = kEmitBytes - 2 * G * (1 + ESZ);
  // stage the 32 encoder tables (8-byte entries), every copy in flight at once
  for (uint32_t k = threadIdx.x; k < kKvTables * 256; k += blockDim.x) {
    const uint32_t t = k >> 8, sidx = k & 255;
    if (SKV_SMEM_OK(t * kEncTabStride + sidx * 8, 8, kSiteSmemStore))
      cp_async_8(t * kEncTabStride + sidx * 8, a.tables + (uint64_t)t * SKV_TABLE_STRIDE + SKV_TABLE_ENC_OFF + sidx * 8);
  }
  cp_async_wait_all();
  // a warp's word buffers double as placement staging slots; its mbarriers
  // follow all the word buffers
  if ((threadIdx.x & 31) < kCpSlots) {
    mbar_init(smem_addr(g_smem) + enc_bars_at(threadIdx.x >> 5, blockDim.x) + 8 * (threadIdx.x & 31), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint32_t tid = threadIdx.x & 31;
  // threads take lanes so that the R lanes sharing a channel set are adjacent:
  // a half-warp's table reads then touch at most 16/R channel sets
  const uint32_t R = 32u * G / a.D, CS = 32u / R;
  const uint32_t lane = (tid % R) * CS + tid / R;
  const uint32_t owner_of_tid = (tid % CS) * R + tid / CS;    // thread coding format lane tid
  const uint32_t buf_top = kEncTabBytes + (threadIdx.x + 1) * kEmitBytes;
  const uint64_t warp_gid = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (warp_gid >= a.slot_warps) return;   // the workspace holds slots for slot_warps warps only
  const uint64_t chunk_pos = (uint64_t)kLanes * a.K;
  // A coded chunk waits in its slot set until the warp has coded the next
  // one; by then its predecessors have published their totals, so placing it
  // rarely waits.
  unsigned long long pend = ~0ull, pend_total = 0;
  uint32_t pend_len = 0, pend_incl = 0, set = 0, phase = 0;
  while (true) {
    unsigned long long chunk = 0;
    if (tid == 0) chunk = atomicAdd(a.ticket, 1ull);
    chunk = __shfl_sync(0xFFFFFFFFu, chunk, 0);
    if (chunk >= a.n_chunks) {
      if (pend != ~0ull)
        place_pending(a, pend, pend_total, pend_len, pend_incl, warp_gid * 2 + (set ^ 1u), CS, R, true, phase);
      break;
    }
    uint8_t* const my_slot_end =
        reinterpret_cast<uint8_t*>(a.slots + ((warp_gid * 2 + set) * kLanes + tid + 1) * a.slot_words);
    const uint64_t slice = chunk / a.cps;
    const uint64_t first = (chunk - slice * a.cps) * chunk_pos;
    const uint64_t n_pos = min(chunk_pos, a.slice_pos - first);
    const uint32_t n_groups = (uint32_t)(n_pos / G);
    const uint32_t n_g = lane < n_groups ? (n_groups - lane + 31) / 32 : 0;
    const int n_iter = (int)((n_groups + 31) / 32);            // warp-uniform (lane 0 has the most)
    // table offsets of the lane's positions: fixed per channel, or (exponent
    // model) recomputed for every group from the base bins bw
    uint32_t tb[G], bw[4];
    if (MODEL) load_lane_bases(a, slice, (lane * G) % a.D, bw);
    else load_lane_tables<ESZ>(a, slice, (lane * G) % a.D, kEncTabStride, tb);
    const uint64_t off = (slice * a.slice_pos + first) * ESZ + lane * 16;
    // byte offset of this lane's group k of the chunk in the caches
    const uint32_t tpi = 32u * G / a.D;   // tokens between a lane's consecutive groups
    const uint64_t tok0 = first / a.D + (lane * G) / a.D;
    const uint32_t d0 = (lane * G) % a.D;
    // paged pools: the block-table entries of groups i - 1 and i - 2 are read
    // while group i is coded (bt1, bt2), so a group load never waits on one
    const uint64_t lk = PAGED ? slice / a.pg.H : 0;
    const uint64_t lkb = PAGED ? (lk * a.pg.n_blocks) << a.pg.shift : 0;
    const uint64_t hd0 = PAGED ? (slice - lk * a.pg.H) * a.D + d0 : 0;
    auto goff = [&](uint32_t k, uint32_t blk) -> uint64_t {
      if (!PAGED) return off + (uint64_t)k * 512;
      bool ok;
      return paged_elem_at(a.pg, blk, tok0 + (uint64_t)k * tpi, lkb, hd0, a.D, a.status, ok) * ESZ;
    };
    auto entry = [&](int k) -> uint32_t {
      return (PAGED && k >= 0) ? paged_entry(a.pg, tok0 + (uint64_t)k * tpi) : 0u;
    };
    uint8_t* gp = my_slot_end;
    uint32_t rp = buf_top;
    uint32_t x = kStateLow;
    uint4 tc = make_uint4(0, 0, 0, 0), pc = tc;
    uint32_t bt1 = 0, bt2 = 0;
    if (n_g) {
      const uint64_t o = goff(n_g - 1, entry((int)n_g - 1));
      tc = ldg_stream(a.tgt + o);
      pc = ldg_stream(a.prd + o);
      bt1 = entry((int)n_g - 2);
      bt2 = entry((int)n_g - 3);
    }
    for (int i = n_iter - 1; i >= 0; --i) {
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, i < (int)n_g);
      if (i >= (int)n_g) continue;
      uint4 tn = tc, pn = pc;
      if (i > 0) {
        const uint64_t o = goff(i - 1, bt1);
        tn = ldg_stream(a.tgt + o);
        pn = ldg_stream(a.prd + o);
      }
      if (PAGED) {
        bt1 = bt2;
        bt2 = entry(i - 3);
      }
      // FP8: word k of the group gives its even bytes in ve[k] and its odd
      // bytes in vo[k] as 16-bit lanes ord(t) + 127 - ord(p), which are the
      // symbols while no position of the group escapes (a negative lane
      // borrows from the next, which only matters when the group escapes).
      // The escape test is on the lane-wise maximum: some lane >= 255
      // exactly when a position needs the escape or a lane went negative.
      // BF16: the symbols of the two halves of each word, tested directly.
      uint32_t ve[4], vo[4];
      bool esc;
      if (ESZ == 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ot = ord8x4(word_of(tc, k)), op = ord8x4(word_of(pc, k));
          uint32_t oto, opo;
          asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(oto) : "r"(ot));
          asm("prmt.b32 %0, %1, 0, 0x4341;" : "=r"(opo) : "r"(op));
          ve[k] = (ot & 0x00FF00FFu) + 0x007F007Fu - (op & 0x00FF00FFu);
          vo[k] = oto + 0x007F007Fu - opo;
        }
        const uint32_t mx = vmax_u16x2(vmax_u16x2(vmax_u16x2(ve[0], vo[0]), vmax_u16x2(ve[1], vo[1])),
                                       vmax_u16x2(vmax_u16x2(ve[2], vo[2]), vmax_u16x2(ve[3], vo[3])));
        esc = ((mx | (mx + 0x00010001u)) & 0xFF00FF00u) != 0u;
      } else {
        uint32_t mx = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ot = ord16x2(word_of(tc, k)), op = ord16x2(word_of(pc, k));
          ve[k] = (ot & 0xFFFFu) + 127u - (op & 0xFFFFu);
          vo[k] = (ot >> 16) + 127u - (op >> 16);
          mx = max(mx, max(ve[k], vo[k]));
        }
        esc = mx > 254u;
      }
      if (ESZ == 2 && !PAGED && __any_sync(act, esc)) {
        // BF16: ve / vo hold the exact residuals + 127 (32-bit lanes); escapes
        // are common enough that the raw steps sit behind a vote per position
        // (the paged variant keeps the path below: its extra registers would spill)
        if (__any_sync(act, buf_top - rp > kRoomEsc)) emit_flush_sync(act, buf_top, rp, gp);
#pragma unroll
        for (int e = G - 1; e >= 0; --e) {
          const uint32_t v = (e & 1) ? vo[e >> 1] : ve[e >> 1];
          const bool e_j = v > 254u;
          if (__any_sync(act, e_j)) {
            const uint32_t raw = (v - 127u) & 0xFFFFu;
            enc_raw_smem_if(x, rp, raw & 0xFFu, e_j);
            enc_raw_smem_if(x, rp, raw >> 8, e_j);
          }
          enc_step_smem(x, rp, lds_u64(tb[e] + (e_j ? 255u : v) * 8u));
        }
      } else if ((ESZ == 1 || PAGED) && __any_sync(act, esc)) {
        // rare: exact residuals per position, raw steps where one escapes
        if (__any_sync(act, buf_top - rp > kRoomEsc)) emit_flush_sync(act, buf_top, rp, gp);
        uint32_t t4[4];
#pragma unroll
        for (int e = G - 1; e >= 0; --e) {
          constexpr uint32_t mk = ESZ == 1 ? 0xFFu : 0xFFFFu;
          const uint32_t sh = ESZ == 1 ? 8 * (e & 3) : 16 * (e & 1);
          const int wi = ESZ == 1 ? (e >> 2) : (e >> 1);
          if (MODEL && (e & 3) == 3) model_exp_word(bw[e >> 2], word_of(pc, e >> 2), kEncTabStride, t4);
          const uint32_t tbe = MODEL ? t4[e & 3] : tb[e];
          const uint32_t ot = ESZ == 1 ? ord8x4(word_of(tc, wi)) : ord16x2(word_of(tc, wi));
          const uint32_t op = ESZ == 1 ? ord8x4(word_of(pc, wi)) : ord16x2(word_of(pc, wi));
          const int r = (int)((ot >> sh) & mk) - (int)((op >> sh) & mk);
          const uint32_t sy = (uint32_t)(r + 127);
          const bool e_j = sy > 254u;
          const uint32_t raw = (uint32_t)r & mk;
          enc_raw_smem_if(x, rp, raw & 0xFFu, e_j);
          if (ESZ == 2) enc_raw_smem_if(x, rp, raw >> 8, e_j);
          enc_step_smem(x, rp, lds_u64(tbe + (e_j ? 255u : sy) * 8u));
        }
      } else {
        if (__any_sync(act, buf_top - rp > kRoomPlain)) emit_flush_sync(act, buf_top, rp, gp);
        uint32_t t4[4];
        // entry of position e: its load is issued two steps before the
        // renormalisation store of the step before it, so the store does not
        // hold the load back
        auto entry_addr = [&](int e) -> uint32_t {
          if (MODEL && (e & 3) == 3) model_exp_word(bw[e >> 2], word_of(pc, e >> 2), kEncTabStride, t4);
          // byte offset of the entry: 8 * symbol (the upper lane's shift
          // also drops the lower lane, whose value is below 2^13)
          const uint32_t tbe = MODEL ? t4[e & 3] : tb[e];
          uint32_t ad;
          if (ESZ == 1) {
            const uint32_t v = (e & 1) ? vo[e >> 2] : ve[e >> 2];
            ad = (e & 2) ? tbe + (v >> 13) : (v & 0xFFFFu) * a.k.k8 + tbe;   // lower lane: multiply-add
          } else {
            ad = tbe + (((e & 1) ? vo[e >> 1] : ve[e >> 1]) << 3);
          }
          SKV_CHECK(ad - tbe < 2048u && tbe + 2048u <= kEncTabBytes, kSiteEncEntry);
          return ad;
        };
        uint2 ent[G];
#pragma unroll
        for (int e = G - 1; e >= G - 2; --e) ent[e] = lds_u64(entry_addr(e));
#pragma unroll
        for (int e = G - 1; e >= 0; --e) {
          if (e - 2 >= 0) ent[e - 2] = lds_u64(entry_addr(e - 2));
          enc_step_smem_fma(x, rp, ent[e], a.k);
        }
      }
      SKV_CHECK(buf_top - rp <= kEmitBytes, kSiteWordBuffer);
      tc = tn;
      pc = pn;
    }
    // room for the two state words, which go out last (read first)
    if (__any_sync(0xFFFFFFFFu, buf_top - rp > kEmitBytes - 4)) emit_flush_sync(0xFFFFFFFFu, buf_top, rp, gp);
    rp -= 2;
    sts_u16(rp, x & 0xFFFFu);
    rp -= 2;
    sts_u16(rp, x >> 16);
    const uint32_t my_bytes = (uint32_t)(my_slot_end - gp) + (buf_top - rp);
    emit_flush_all(buf_top, rp, gp);
    SKV_CHECK((uint64_t)(my_slot_end - gp) <= 2 * a.slot_words, kSiteScratchSlot);
    // lane lengths in format-lane order and the chunk total
    const uint32_t len = __shfl_sync(0xFFFFFFFFu, my_bytes, owner_of_tid);
    uint32_t incl = len;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (tid >= (uint32_t)o) incl += u;
    }
    const unsigned long long total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    chunk_publish(a.chunk_state, chunk, total);
    if (pend != ~0ull) {
      phase = place_pending(a, pend, pend_total, pend_len, pend_incl, warp_gid * 2 + (set ^ 1u), CS, R,
                            chunk >= a.last_wave, phase);
      if (phase & kPlaceFailed) return;   // flagged; the warp's copies are waited for
    }
    pend = chunk;
    pend_total = total;
    pend_len = len;
    pend_incl = incl;
    set ^= 1u;
  }
}

// Self-test of the encoder's bounded wait: warp w plays chunk w (total w + 1
// bytes) through chunk_lookback; chunk `missing` never publishes, so its
// successors must give up after max_spins polls and report a timeout.
__global__ void k_selftest_lookback(unsigned long long* st, uint32_t n, uint32_t missing, uint32_t max_spins,
                                    uint32_t* status, unsigned long long* excl_out) {
  const uint32_t w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= n || w == missing) return;
  const unsigned long long e = chunk_lookback(st, w, w + 1, status, max_spins);
  if ((threadIdx.x & 31) == 0) excl_out[w] = e;
}

// ---------------------------------------------------------------------------
// Decoder, KV caches, fused with reconstruction.  Each lane reads its words
// through a shared-memory ring (refilled once per FP8 group on the speculative
// pass, every SUB symbols where escapes are decoded), looks the slot
// up in the shared slot->symbol table, rebuilds the target from the
// prediction's ordinal and stores whole 16-byte groups.
// ---------------------------------------------------------------------------
// Decode one position exactly (escapes included) and add its symbol term to
// the packed word sw: for a plain symbol the term is sym << sh, for an escape
// it is (t - p + 127) << sh with t = (p + raw) mod 2^W, so that in every case
// ord(target word) = ord(prediction word) + sw - 127 per element, exactly.
template <int ESZ>
__device__ __forceinline__ void dec_exact(RingLane& L, uint32_t tbe, uint32_t pwd, uint32_t sh, uint32_t act,
                                          uint32_t& sw) {
  constexpr uint32_t mk = ESZ == 1 ? 0xFFu : 0xFFFFu;
  const uint32_t slot = L.x & 4095u;
  const uint32_t sym = lds_u8(tbe + slot);
  const uint32_t dv = lds_u32(tbe + 4096u + sym * 4u);
  L.x = (dv & 0xFFFFu) * (L.x >> 12) + slot + (uint32_t)((int32_t)dv >> 16);   // + (-cum)
  ring_renorm(L);
  uint32_t term = sym;
  // escapes are rare: a warp-uniform test keeps their steps off the common
  // path; inside, the raw steps are predicated per lane (no nested branch)
  if (__any_sync(act, sym == 255u)) {
    const bool esc = sym == 255u;
    uint32_t v = ring_raw_if(L, esc);
    if (ESZ == 2) v = (v << 8) | ring_raw_if(L, esc);
    const uint32_t pe = (pwd >> sh) & mk;
    term = esc ? ((pe + v) & mk) - pe + 127u : sym;
  }
  sw += term << sh;
}

template <int ESZ, bool PAGED, bool MODEL>
__global__ void __launch_bounds__(dec_threads(PAGED, MODEL), 1) k_decode_kv(CodecArgs a) {
  constexpr int G = 16 / ESZ;
  constexpr int SUB = ESZ == 1 ? 8 : 4;   // at most 32 / 24 stream bytes between refills
  constexpr uint32_t kBias = ESZ == 1 ? 0x7F7F7F7Fu : 0x007F007Fu;
  // stage the 32 slot->symbol + decoder tables, every copy in flight at once
  for (uint32_t k = threadIdx.x; k < kKvTables * 1280; k += blockDim.x) {
    const uint32_t t = k / 1280, w = k % 1280;
    if (SKV_SMEM_OK(t * kDecTabStride + 4 * w, 4, kSiteSmemStore))
      cp_async_4(t * kDecTabStride + 4 * w, a.tables + (uint64_t)t * SKV_TABLE_STRIDE + SKV_TABLE_LUT_OFF + 4 * w);
  }
  cp_async_wait_all();
  __syncthreads();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t ring = kDecTabBytes + threadIdx.x * kRingStride;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint64_t chunk_pos = (uint64_t)kLanes * a.K;
  for (uint64_t chunk = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); chunk < a.n_chunks;
       chunk += warps) {
    const uint64_t slice = chunk / a.cps;
    const uint64_t first = (chunk - slice * a.cps) * chunk_pos;
    const uint64_t n_pos = min(chunk_pos, a.slice_pos - first);
    const uint32_t n_groups = (uint32_t)(n_pos / G);
    const uint32_t n_g = lane < n_groups ? (n_groups - lane + 31) / 32 : 0;
    uint32_t tb[G], bw[4];
    if (MODEL) load_lane_bases(a, slice, (lane * G) % a.D, bw);
    else load_lane_tables<ESZ>(a, slice, (lane * G) % a.D, kDecTabStride, tb);
    const uint64_t g = chunk * kLanes + lane;
    uint64_t sa, sb;
    const bool ok = lane_span(a.offs, g, a.n_lanes, a.n_bytes, &sa, &sb);
    RingLane L;
    ring_open(L, a.bs, ring, sa, sb, ok, a.status);
    const uint64_t off = (slice * a.slice_pos + first) * ESZ + lane * 16;
    // byte offset of this lane's group k of the chunk in the caches (ok: the
    // paged block-table entry is in range)
    const uint32_t tpi = 32u * G / a.D;
    const uint64_t tok0 = first / a.D + (lane * G) / a.D;
    const uint32_t d0 = (lane * G) % a.D;
    // paged pools: entries of groups i + 1 and i + 2 are read ahead (btn1, btn2)
    const uint64_t lk = PAGED ? slice / a.pg.H : 0;
    const uint64_t lkb = PAGED ? (lk * a.pg.n_blocks) << a.pg.shift : 0;
    const uint64_t hd0 = PAGED ? (slice - lk * a.pg.H) * a.D + d0 : 0;
    auto goff = [&](uint32_t k, uint32_t blk, bool& ok) -> uint64_t {
      ok = true;
      if (!PAGED) return off + (uint64_t)k * 512;
      return paged_elem_at(a.pg, blk, tok0 + (uint64_t)k * tpi, lkb, hd0, a.D, a.status, ok) * ESZ;
    };
    auto entry = [&](uint32_t k) -> uint32_t {
      return (PAGED && k < n_g) ? paged_entry(a.pg, tok0 + (uint64_t)k * tpi) : 0u;
    };
    uint4 pc = make_uint4(0, 0, 0, 0);
    uint32_t btc = entry(0), btn1 = entry(1), btn2 = entry(2);
    if (n_g) {
      bool ok;
      pc = ldg_stream(a.prd + goff(0, btc, ok));
    }
    const uint32_t n_iter = (n_groups + 31) / 32;              // warp-uniform
    for (uint32_t i = 0; i < n_iter; ++i) {
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, i < n_g);
      if (i >= n_g) continue;
      uint4 pn = pc;
      if (i + 1 < n_g) {
        bool ok;
        pn = ldg_stream(a.prd + goff(i + 1, btn1, ok));
      }
      if (MODEL) model_exp_tables(bw, pc, kDecTabStride, tb);
      uint32_t pw[4], sw[4] = {0, 0, 0, 0};
#pragma unroll
      for (int k = 0; k < 4; ++k) pw[k] = ESZ == 1 ? ord8x4(word_of(pc, k)) : ord16x2(word_of(pc, k));
      if (ESZ == 1) {
        // FP8: the group's 16 positions are decoded assuming no escape; if
        // any lane met one, those lanes decode the group again from the saved
        // state (ring reloaded from the stream) with escapes handled.  Without
        // raw steps a position consumes at most one word, so the 16 positions
        // read at most 32 bytes: one refill at the group's start keeps the
        // ring ahead of them.
        const uint32_t x0 = L.x, p0 = L.p;
        bool esc = false;
#pragma unroll
        for (int e = 0; e < G; ++e) {
          if (e == 0) ring_refill(L, act);
          const uint32_t slot = L.x & 4095u;
          const uint32_t sym = lds_u8(tb[e] + slot);
          const uint32_t dv = lds_u32(tb[e] + 4096u + sym * 4u);
          L.x = (dv & 0xFFFFu) * (L.x >> 12) + slot + (uint32_t)((int32_t)dv >> 16);   // + (-cum)
          ring_renorm(L);
          esc |= sym == 255u;
          sw[e >> 2] += sym << (8 * (e & 3));
        }
        const uint32_t redo = __ballot_sync(act, esc);
        if (redo) {
          if (esc) {
            ring_reopen(L, p0);
            L.x = x0;
            L.nxt = ring_word(L, p0);   // the word at p0, reloaded with the ring
            sw[0] = sw[1] = sw[2] = sw[3] = 0;
#pragma unroll
            for (int e = 0; e < G; ++e) {
              if (e % SUB == 0 && e) ring_refill(L, redo);
              dec_exact<ESZ>(L, tb[e], pw[e >> 2], 8 * (e & 3), redo, sw[e >> 2]);
            }
          }
          __syncwarp(act);
        }
      } else {
#pragma unroll
        for (int e = 0; e < G; ++e) {
          if (e % SUB == 0) ring_refill(L, act);
          dec_exact<ESZ>(L, tb[e], pw[e >> 1], 16 * (e & 1), act, sw[e >> 1]);
        }
      }
      // ord(target) = ord(prediction) + sw - 127 per element, exact as a
      // plain 32-bit sum (every element's result lies in its own field)
      uint4 o;
      o.x = ESZ == 1 ? unord8x4(pw[0] + sw[0] - kBias) : unord16x2(pw[0] + sw[0] - kBias);
      o.y = ESZ == 1 ? unord8x4(pw[1] + sw[1] - kBias) : unord16x2(pw[1] + sw[1] - kBias);
      o.z = ESZ == 1 ? unord8x4(pw[2] + sw[2] - kBias) : unord16x2(pw[2] + sw[2] - kBias);
      o.w = ESZ == 1 ? unord8x4(pw[3] + sw[3] - kBias) : unord16x2(pw[3] + sw[3] - kBias);
      bool ok;
      const uint64_t oo = goff(i, btc, ok);
      SKV_CHECK(PAGED || oo + 16 <= (a.n_chunks / a.cps) * a.slice_pos * ESZ, kSiteDecOut);
      if (ok) stg_stream(a.out + oo, o);
      pc = pn;
      if (PAGED) {
        btc = btn1;
        btn1 = btn2;
        btn2 = entry(i + 3);
      }
    }
    ring_close(L, a.status);
  }
}

// ---------------------------------------------------------------------------
// Transform-coefficient streams (int16 q, fp32 mean mu, 1024 tables).
// Positions are the full [token][coef] grid; switched-off components carry
// no symbol.  Tables are read through the cache hierarchy.
// ---------------------------------------------------------------------------
// mu -> (m, f): mu rounded to the nearest 1/16 (ties up) in fp32,
// m = floor(mu_q / 16), f = mu_q mod 16
__device__ __forceinline__ void coef_mean(float mu, int* m, uint32_t* f) {
  const float t = __fadd_rn(__fmul_rn(mu, 16.0f), 0.5f);
  const int mq = fabsf(t) < 67108864.0f ? (int)floorf(t) : 0;
  *m = mq >> 4;
  *f = (uint32_t)mq & 15u;
}

// The 8 positions of a group: q and mu as read from memory (vectors when the
// group is whole; loaded one group ahead of their use), then per position the
// mean split, the table and whether the position is coded (skip: components
// switched off, bin 0xFF, and positions past the slice end).
struct CoefRaw {
  float4 m0, m1;
  uint4 q;
};
struct CoefGroup {
  int m[8];
  uint32_t tbl[8];
  int16_t q[8];
  uint32_t skip;
};
__device__ __forceinline__ void coef_load(const CodecArgs& a, uint64_t p0, uint32_t ne, bool with_q, CoefRaw& R) {
  const int16_t* q = reinterpret_cast<const int16_t*>(a.tgt);
  const float* mu = reinterpret_cast<const float*>(a.prd);
  if (ne == 8) {
    // streaming loads: read once, so that they do not push the tables out of L2
    R.m0 = __ldcs(reinterpret_cast<const float4*>(mu + p0));
    R.m1 = __ldcs(reinterpret_cast<const float4*>(mu + p0) + 1);
    R.q = with_q ? __ldcs(reinterpret_cast<const uint4*>(q + p0)) : make_uint4(0, 0, 0, 0);
    return;
  }
  float mv[8];
  uint32_t qw[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mv[e] = (uint32_t)e < ne ? __ldg(mu + p0 + e) : 0.f;
    if (with_q && (uint32_t)e < ne) qw[e >> 1] |= (uint32_t)(uint16_t)__ldg(q + p0 + e) << (16 * (e & 1));
  }
  R.m0 = make_float4(mv[0], mv[1], mv[2], mv[3]);
  R.m1 = make_float4(mv[4], mv[5], mv[6], mv[7]);
  R.q = make_uint4(qw[0], qw[1], qw[2], qw[3]);
}
// c = the component of the group's first position (callers step it from
// group to group: no 64-bit remainder per group).  A whole group whose
// components do not wrap reads its 8 bins as one 8-byte vector.
__device__ __forceinline__ void coef_group(const CodecArgs& a, uint32_t c, uint32_t ne, const CoefRaw& R,
                                           CoefGroup& G) {
  const float mv[8] = {R.m0.x, R.m0.y, R.m0.z, R.m0.w, R.m1.x, R.m1.y, R.m1.z, R.m1.w};
  const uint32_t qw[4] = {R.q.x, R.q.y, R.q.z, R.q.w};
  uint32_t bins[8];
  if (ne == 8 && c + 8 <= a.C && (c & 7u) == 0) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.bins + c));
#pragma unroll
    for (int e = 0; e < 8; ++e) bins[e] = ((e < 4 ? v.x : v.y) >> (8 * (e & 3))) & 0xFFu;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bins[e] = (uint32_t)e < ne ? __ldg(a.bins + c) : 0xFFu;
      c = c + 1 == a.C ? 0 : c + 1;
    }
  }
  G.skip = 0;
  bool bad = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    G.q[e] = (int16_t)(qw[e >> 1] >> (16 * (e & 1)));
    uint32_t f;
    coef_mean(mv[e], &G.m[e], &f);
    const uint32_t bin = bins[e];
    G.skip |= (bin == 0xFFu ? 1u : 0u) << e;
    bad |= bin > 63u && bin != 0xFFu;
    G.tbl[e] = 16u * min(bin, 63u) + f;   // a skipped component's table is never read
    SKV_CHECK(G.tbl[e] < kCoefTables, kSiteCoefTable);
  }
  if (bad) atomicOr(a.status, SKV_FLAG_BAD_BIN);
}
// component of the previous / next group of a lane (groups 256 positions apart)
__device__ __forceinline__ uint32_t coef_comp_back(uint32_t c, uint32_t step, uint32_t C) {
  return c >= step ? c - step : c + C - step;
}
__device__ __forceinline__ uint32_t coef_comp_fwd(uint32_t c, uint32_t step, uint32_t C) {
  const uint32_t n = c + step;
  return n >= C ? n - C : n;
}

// One coding step where do_it holds; elsewhere x and the stream are left alone
// (the entry must still be a valid one: the step is computed, then dropped).
__device__ __forceinline__ void enc_step_gmem_if(uint32_t& x, uint16_t*& wp, uint2 e, bool do_it) {
  const bool ren = do_it && x >= (e.y & 0xFFF00000u);
  if (ren) *(wp - 1) = (uint16_t)x;
  wp -= ren ? 1 : 0;
  const uint32_t xr = ren ? x >> 16 : x;
  const uint32_t q = enc_quot(xr, e.x, e.y);
  const uint32_t xn = xr + q * (4096u - (e.y >> 20)) + ((e.y >> 8) & 0xFFFu);
  x = do_it ? xn : x;
}

// Groups of 8 positions go to the lanes in turn (group g of a chunk to lane
// g mod 32).  A group's inputs are read one group ahead; its 8 table entries
// are fetched before its steps so that their loads overlap.  Escapes take a
// warp-uniform branch.  (Fetching the entries one group ahead as well, so that
// their latency overlaps the previous group's steps, measured slower.)
__global__ void __launch_bounds__(256) k_encode_coef(CodecArgs a) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint64_t chunk_pos = (uint64_t)kLanes * a.K;
  const uint2* const encb = reinterpret_cast<const uint2*>(a.tables + SKV_TABLE_ENC_OFF);
  constexpr uint32_t kEntStride = SKV_TABLE_STRIDE / 8;
  for (uint64_t chunk = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); chunk < a.n_chunks;
       chunk += warps) {
    const uint64_t first = chunk * chunk_pos;
    const uint64_t n_pos = min(chunk_pos, a.slice_pos - first);
    const uint32_t n_groups = (uint32_t)((n_pos + 7) / 8);
    const uint32_t n_g = lane < n_groups ? (n_groups - lane + 31) / 32 : 0;
    const int n_iter = (int)((n_groups + 31) / 32);            // warp-uniform (lane 0 has the most)
    const uint64_t g = chunk * kLanes + lane;
    uint16_t* const slot_end = a.slots + (g + 1) * a.slot_words;
    uint16_t* wp = slot_end;
    uint32_t x = kStateLow;
    auto gpos = [&](int i) { return first + ((uint64_t)i * 32 + lane) * 8; };   // position of group i
    auto gnum = [&](uint64_t p0) { return (uint32_t)min((uint64_t)8, first + n_pos - p0); };
    CoefRaw R;
    const uint32_t step = 256u % a.C;
    uint32_t comp = n_g ? (uint32_t)(gpos((int)n_g - 1) % a.C) : 0u;   // component of the lane's current group
    if (n_g) coef_load(a, gpos((int)n_g - 1), gnum(gpos((int)n_g - 1)), true, R);
    for (int i = n_iter - 1; i >= 0; --i) {
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, i < (int)n_g);
      if (i >= (int)n_g) continue;
      const uint64_t p0 = gpos(i);
      const uint32_t ne = gnum(p0);
      CoefGroup G;
      coef_group(a, comp, ne, R, G);
      comp = coef_comp_back(comp, step, a.C);
      if (i > 0) coef_load(a, gpos(i - 1), gnum(gpos(i - 1)), true, R);
      uint2 en[8];
      uint32_t esc = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool d = !((G.skip >> e) & 1u);
        uint32_t sym = (uint32_t)((int)G.q[e] - G.m[e] + 127);
        if (sym > 254u) {
          sym = 255;
          esc |= (d ? 1u : 0u) << e;
        }
        en[e] = __ldg(encb + (d ? G.tbl[e] : 0u) * kEntStride + sym);
      }
      if (__any_sync(act, esc != 0)) {
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          if ((esc >> e) & 1u) {
            const uint32_t raw = (uint32_t)((int)G.q[e] - G.m[e]) & 0xFFFFu;
            enc_raw_gmem(x, wp, raw & 0xFFu);
            enc_raw_gmem(x, wp, raw >> 8);
          }
          enc_step_gmem_if(x, wp, en[e], !((G.skip >> e) & 1u));
        }
      } else {
#pragma unroll
        for (int e = 7; e >= 0; --e) enc_step_gmem_if(x, wp, en[e], !((G.skip >> e) & 1u));
      }
    }
    *--wp = (uint16_t)x;
    *--wp = (uint16_t)(x >> 16);
    a.lane_words[g] = (uint32_t)(slot_end - wp);
  }
}

// Decoding reads one slot entry per step (symbol, frequency and offset: see
// the table layout), a dependent L2 read: the step chain is bound by its latency,
// so nothing else sits between two reads of a lane (escapes are handled by
// redoing the group).
__global__ void __launch_bounds__(256) k_decode_coef(CodecArgs a) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  const uint64_t chunk_pos = (uint64_t)kLanes * a.K;
  int16_t* q = reinterpret_cast<int16_t*>(a.out);
  const uint32_t* slot_tab = reinterpret_cast<const uint32_t*>(a.tables + (uint64_t)kCoefTables * SKV_TABLE_STRIDE);
  for (uint64_t chunk = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); chunk < a.n_chunks;
       chunk += warps) {
    const uint64_t first = chunk * chunk_pos;
    const uint64_t n_pos = min(chunk_pos, a.slice_pos - first);
    const uint32_t n_groups = (uint32_t)((n_pos + 7) / 8);
    const uint32_t n_g = lane < n_groups ? (n_groups - lane + 31) / 32 : 0;
    const uint32_t n_iter = (n_groups + 31) / 32;              // warp-uniform
    const uint64_t g = chunk * kLanes + lane;
    uint64_t sa, sb;
    const bool ok = lane_span(a.offs, g, a.n_lanes, a.n_bytes, &sa, &sb);
    DecLane L;
    dec_open(L, a.bs, sa, sb, ok, a.status);
    auto gpos = [&](uint32_t i) { return first + ((uint64_t)i * 32 + lane) * 8; };
    auto gnum = [&](uint64_t p0) { return (uint32_t)min((uint64_t)8, first + n_pos - p0); };
    CoefRaw R;
    const uint32_t step = 256u % a.C;
    uint32_t comp = n_g ? (uint32_t)(gpos(0) % a.C) : 0u;   // component of the lane's current group
    if (n_g) coef_load(a, gpos(0), gnum(gpos(0)), false, R);
    for (uint32_t i = 0; i < n_iter; ++i) {
      const uint32_t act = __ballot_sync(0xFFFFFFFFu, i < n_g);
      if (i >= n_g) continue;
      const uint64_t p0 = gpos(i);
      const uint32_t ne = gnum(p0);
      CoefGroup G;
      coef_group(a, comp, ne, R, G);
      comp = coef_comp_fwd(comp, step, a.C);
      if (i + 1 < n_g) coef_load(a, gpos(i + 1), gnum(gpos(i + 1)), false, R);
      // The group is decoded assuming no escape (no vote between the dependent
      // table reads); lanes that met one decode it again from the saved state
      // with the raw steps.
      uint32_t qo[4] = {0, 0, 0, 0};
      const uint32_t x0 = L.x, p0w = L.p, n0 = L.nxt;
      bool esc = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool d = !((G.skip >> e) & 1u);
        const uint32_t se = __ldg(slot_tab + (d ? G.tbl[e] : 0u) * 4096u + (L.x & 4095u));
        const uint32_t sym = se & 0xFFu;
        const uint32_t xn = ((se >> 8) & 0xFFFu) * (L.x >> 12) + (se >> 20);
        L.x = d ? xn : L.x;
        dec_renorm(L);                    // a skipped position leaves x >= 2^16: no renormalisation
        esc |= d && sym == 255u;
        qo[e >> 1] |= (d ? (((uint32_t)G.m[e] + sym - 127u) & 0xFFFFu) : 0u) << (16 * (e & 1));
      }
      const uint32_t redo = __ballot_sync(act, esc);
      if (redo) {
        if (esc) {
          L.x = x0;
          L.p = p0w;
          L.nxt = n0;
          qo[0] = qo[1] = qo[2] = qo[3] = 0;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool d = !((G.skip >> e) & 1u);
            const uint32_t se = __ldg(slot_tab + (d ? G.tbl[e] : 0u) * 4096u + (L.x & 4095u));
            const uint32_t sym = se & 0xFFu;
            const uint32_t xn = ((se >> 8) & 0xFFFu) * (L.x >> 12) + (se >> 20);
            L.x = d ? xn : L.x;
            dec_renorm(L);
            uint32_t r = (uint32_t)((int)sym - 127);
            if (__any_sync(redo, d && sym == 255u)) {
              if (d && sym == 255u) {
                r = dec_raw(L);
                r = (r << 8) | dec_raw(L);
              }
            }
            qo[e >> 1] |= (d ? (((uint32_t)G.m[e] + r) & 0xFFFFu) : 0u) << (16 * (e & 1));
          }
        }
        __syncwarp(act);
      }
      if (ne == 8) {
        *reinterpret_cast<uint4*>(q + p0) = make_uint4(qo[0], qo[1], qo[2], qo[3]);
      } else {
#pragma unroll
        for (uint32_t e = 0; e < 8; ++e)
          if (e < ne) q[p0 + e] = (int16_t)(qo[e >> 1] >> (16 * (e & 1)));
      }
    }
    dec_close(L, a.status);
  }
}

// ---------------------------------------------------------------------------
// Checkerboard context ([DCKV] how it differs): the means of the odd token
// rows of a coefficient stream from the decoded even rows on both sides,
// through a rank-R linear map with int8 factors V [R][C], U [C][R]:
//   x = clamp(q_even[t] + q_even[t + 1], +-127)
//   g = clamp(floor(V x / 2^s1), +-127),   k = floor(U g / 2^s2)
//   mu' = clamp(mu_q + k, +-(2^23 - 1)) / 16   (mu_q: the mean quantisation)
// The map's entries are used clamped to [-8, 8] (4-bit weights kept in int8).
// Both products run on the tensor cores in bf16 with fp32 accumulation and
// are exact: operands are small integers (|x|, |g| <= 127, |w| <= 8) and
// every partial sum stays below K * 127 * 8 < 2^24 for K <= 16384 (checked on
// the host), so any summation order gives the same integer.
// ---------------------------------------------------------------------------
constexpr uint32_t kUmBM = 128, kUmBK = 64;   // output tile rows and k-block (64 bf16 = 128 B rows)
constexpr uint32_t kUmBN = 128;                              // output tile columns
constexpr uint32_t kUmStages = 3;                            // k-blocks in flight
constexpr uint32_t kUmCtas = 2;                              // CTAs per SM (one's epilogue overlaps the other's MMAs)
constexpr uint32_t kUmThreads = 512;                         // 16 warps: four per tensor-memory lane quarter
constexpr uint32_t kUmTileA = kUmBM * kUmBK * 2, kUmTileB = kUmBN * kUmBK * 2;
constexpr uint32_t kUmStage = kUmTileA + kUmTileB;
constexpr uint32_t kUmOutPitch = kUmBN + 4;                  // staged output row (32-bit words)
static_assert(kUmBM * kUmOutPitch * 4 <= kUmStages * kUmStage, "output staging fits in the stages");
constexpr uint32_t kUmSmem = kUmStages * kUmStage + 1024 + 256;
// instruction descriptor (kind::f16): fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N / 8 at bit 17, M / 16 at bit 24
constexpr uint32_t kUmIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kUmBN >> 3) << 17) | ((kUmBM >> 4) << 24);

// 2-D tile load (x = inner element index, y = row) completing on `bar`
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, uint32_t x, uint32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// shared-memory matrix descriptor: K-major rows of 128 B in the 128-byte
// swizzle (the layout the tile loads write), 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem, uint64_t da, uint64_t db, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          tmem),
      "l"(da), "l"(db), "r"(kUmIdesc), "r"(accumulate));
}
// arrive on `bar` once every earlier tcgen05.mma of this thread has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of the warp's 32 accumulator rows (one row per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// x rows as bf16: block t builds row t, eight coefficients per thread and step
__global__ void __launch_bounds__(256) k_ctx_x(const int16_t* qe, uint64_t n_even, uint32_t C, __nv_bfloat16* X) {
  const uint64_t t = blockIdx.x;
  const bool next = t + 1 < n_even;
  const int16_t* r0 = qe + t * C;
  const int16_t* r1 = r0 + C;
  __nv_bfloat16* xr = X + t * C;
  for (uint32_t j = threadIdx.x * 8; j < C; j += blockDim.x * 8) {
    const uint4 a = *reinterpret_cast<const uint4*>(r0 + j);
    const uint4 b = next ? *reinterpret_cast<const uint4*>(r1 + j) : make_uint4(0, 0, 0, 0);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int lo = (int)(int16_t)(aw[k] & 0xFFFFu) + (int)(int16_t)(bw[k] & 0xFFFFu);
      int hi = (int)(int16_t)(aw[k] >> 16) + (int)(int16_t)(bw[k] >> 16);
      lo = lo < -127 ? -127 : (lo > 127 ? 127 : lo);
      hi = hi < -127 ? -127 : (hi > 127 ? 127 : hi);
      const __nv_bfloat162 h = __halves2bfloat162(__int2bfloat16_rn(lo), __int2bfloat16_rn(hi));
      o[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(xr + j) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}
// map factor entries, clamped to [-8, 8], as bf16 operands
__global__ void __launch_bounds__(256) k_ctx_w(const int8_t* w, uint64_t n, __nv_bfloat16* wb) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int v = w[i];
  v = v < -8 ? -8 : (v > 8 ? 8 : v);
  wb[i] = __int2bfloat16_rn(v);
}

// Out[M][N] = epilogue(A[M][K] . B[N][K]^T), A and B bf16 row-major (K-major),
// one 128 x kUmBN output tile per CTA on the 5th-generation tensor cores:
// thread 0 streams k-blocks of both operands into a ring of shared-memory
// stages with tile loads, thread 32 issues the MMAs into a 128 x kUmBN fp32
// accumulator in tensor memory and releases each stage when its MMAs
// complete.  The sixteen warps then move the accumulator (warp w: rows
// 32 (w mod 4).., its tensor-memory lane quarter, 32 columns from 32 (w / 4))
// through shared memory, as floor(acc / 2^s), so that each row of the output
// is written (and, EPI 1, mu read) by a whole warp at once.
// Rows past M and k past K load as zeros.
// EPI 0: G = bf16(clamp(floor(acc / 2^s), +-127));  EPI 1: mu' from mu and
// floor(acc / 2^s).  N is a multiple of 32 (checked on the host).
template <int EPI>
__global__ void __launch_bounds__(kUmThreads, kUmCtas) k_ctx_umma(const __grid_constant__ CUtensorMap tmA,
                                                           const __grid_constant__ CUtensorMap tmB, uint32_t M,
                                                           uint32_t N, uint32_t K, uint32_t s, __nv_bfloat16* G,
                                                           const float* mu, float* out, uint32_t* status,
                                                           uint32_t no_loads) {
  const uint32_t base = (smem_addr(g_smem) + 1023u) & ~1023u;   // stages need 1024-byte alignment
  const uint32_t bar_full = base + kUmStages * kUmStage;
  const uint32_t bar_empty = bar_full + 8 * kUmStages;
  const uint32_t bar_done = bar_empty + 8 * kUmStages;
  const uint32_t tslot = bar_done + 8;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t m0 = blockIdx.y * kUmBM, n0 = blockIdx.x * kUmBN;
  const uint32_t nk = (K + kUmBK - 1) / kUmBK;
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < kUmStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, 1);
    }
    mbar_init(bar_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(kUmBN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(tslot) : "memory");
  bool ok = true;
  if (threadIdx.x == 0 && !no_loads) {   // no_loads: self-test of the bounded waits (nothing arrives)
    for (uint32_t kb = 0; kb < nk; ++kb) {
      const uint32_t st = kb % kUmStages;
      if (kb >= kUmStages && !mbar_wait(bar_empty + 8 * st, ((kb / kUmStages) - 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t dst = base + st * kUmStage;
      mbar_expect_tx(bar_full + 8 * st, kUmStage);
      tma_load_2d(dst, &tmA, kb * kUmBK, m0, bar_full + 8 * st);
      tma_load_2d(dst + kUmTileA, &tmB, kb * kUmBK, n0, bar_full + 8 * st);
    }
  } else if (threadIdx.x == 32) {
    for (uint32_t kb = 0; kb < nk; ++kb) {
      const uint32_t st = kb % kUmStages;
      if (!mbar_wait(bar_full + 8 * st, (kb / kUmStages) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = umma_desc(base + st * kUmStage), db = umma_desc(base + st * kUmStage + kUmTileA);
#pragma unroll
      for (uint32_t k = 0; k < kUmBK / 16; ++k)        // 16 bf16 = 32 bytes along the swizzled row
        umma_bf16(tmem, da + 2 * k, db + 2 * k, (kb | k) != 0);
      umma_commit(bar_empty + 8 * st);
    }
    umma_commit(bar_done);
  }
  __syncwarp();
  bool done = mbar_wait(bar_done, 0);
  if (!done) ok = false;
  tc_fence_after();
  // a wait that ran out anywhere in the CTA: the accumulator is not read and
  // nothing is stored (the output is undefined; SKV_FLAG_TIMEOUT is set)
  const bool failed = __syncthreads_or(!ok) != 0;
  // accumulator rows -> floor(acc / 2^s) in the (now idle) stages, row r at r * kUmOutPitch words;
  // warp w reads rows 32 (w mod 4) .. (its tensor-memory lane quarter), columns of part w / 4
  constexpr uint32_t kParts = kUmThreads / 128, kPartCols = kUmBN / kParts;
  const uint32_t q4 = warp & 3, part = warp >> 2;
  const uint32_t srow = base + (q4 * 32 + lane) * kUmOutPitch * 4;
#pragma unroll 1
  for (uint32_t c0 = part * kPartCols; !failed && c0 < (part + 1) * kPartCols; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tmem + ((q4 * 32u) << 16) + c0, r);
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const int v0 = (int)__uint_as_float(r[j]) >> s, v1 = (int)__uint_as_float(r[j + 1]) >> s;
      const int v2 = (int)__uint_as_float(r[j + 2]) >> s, v3 = (int)__uint_as_float(r[j + 3]) >> s;
      asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(srow + (c0 + j) * 4), "r"(v0), "r"(v1), "r"(v2),
                   "r"(v3)
                   : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  // tensor memory is freed once every MMA has completed (a second bounded wait if the first ran out)
  if (warp == 2) {
    if (!done) done = mbar_wait(bar_done, 0);
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kUmBN));
  }
  if (failed) {
    if (threadIdx.x == 0) atomicOr(status, SKV_FLAG_TIMEOUT);
    return;
  }
  // rows out: warp w takes rows w, w + 8, ...; lane l columns 4l..4l+3 (+128);
  // eight rows per step, so that their mu loads are in flight together
  constexpr uint32_t kRows = 8, kWarps = kUmThreads / 32;
#pragma unroll 1
  for (uint32_t r0 = warp; r0 < kUmBM; r0 += kWarps * kRows) {
#pragma unroll
    for (uint32_t c = lane * 4; c < kUmBN; c += 128) {
      const uint32_t n = n0 + c;
      if (n >= N) continue;
      float4 m4[kRows];
      if (EPI == 1) {
#pragma unroll
        for (uint32_t i = 0; i < kRows; ++i) {
          const uint32_t row = m0 + r0 + kWarps * i;
          m4[i] = row < M ? *reinterpret_cast<const float4*>(mu + (uint64_t)row * N + n) : make_float4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (uint32_t i = 0; i < kRows; ++i) {
        const uint32_t rr = r0 + kWarps * i, row = m0 + rr;
        if (row >= M) continue;
        int v[4];
        asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                     : "r"(base + (rr * kUmOutPitch + c) * 4)
                     : "memory");
        const uint64_t o = (uint64_t)row * N + n;
        if (EPI == 0) {
          int w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) w[u] = v[u] < -127 ? -127 : (v[u] > 127 ? 127 : v[u]);
          const __nv_bfloat162 h0 = __halves2bfloat162(__int2bfloat16_rn(w[0]), __int2bfloat16_rn(w[1]));
          const __nv_bfloat162 h1 = __halves2bfloat162(__int2bfloat16_rn(w[2]), __int2bfloat16_rn(w[3]));
          *reinterpret_cast<uint2*>(G + o) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
        } else {
          const float mv[4] = {m4[i].x, m4[i].y, m4[i].z, m4[i].w};
          float res[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            int mm;
            uint32_t ff;
            coef_mean(mv[u], &mm, &ff);
            int q = 16 * mm + (int)ff + v[u];      // |16 mm + ff| < 2^26, |v| < 2^24: no overflow
            q = q < -8388607 ? -8388607 : (q > 8388607 ? 8388607 : q);
            res[u] = (float)q * 0.0625f;
          }
          *reinterpret_cast<float4*>(out + o) = make_float4(res[0], res[1], res[2], res[3]);
        }
      }
    }
  }
  if (!ok) atomicOr(status, SKV_FLAG_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Lane lengths -> byte offsets: three-phase exclusive scan, then compaction.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_scan_reduce(const uint32_t* lw, uint64_t n,
                                                     unsigned long long* part) {
  __shared__ unsigned long long red[8];
  const uint64_t b0 = (uint64_t)blockIdx.x * kScanPerBlock;
  unsigned long long s = 0;
  for (uint32_t k = threadIdx.x; k < kScanPerBlock; k += 256) {
    const uint64_t i = b0 + k;
    if (i < n) s += lw[i];
  }
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int k = 0; k < 8; ++k) t += red[k];
    part[blockIdx.x] = t;
  }
}

// exclusive scan of part[0..nb) in place; single CTA of 1024 threads
__global__ void __launch_bounds__(1024) k_scan_parts(unsigned long long* part, uint64_t nb) {
  __shared__ unsigned long long wsum[32];
  __shared__ unsigned long long carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (uint64_t base = 0; base < nb; base += 1024) {
    const uint64_t i = base + threadIdx.x;
    const unsigned long long v = i < nb ? part[i] : 0;
    unsigned long long incl = v;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if ((threadIdx.x & 31) >= (uint32_t)o) incl += u;
    }
    if ((threadIdx.x & 31) == 31) wsum[threadIdx.x >> 5] = incl;
    __syncthreads();
    if (threadIdx.x < 32) {
      unsigned long long w = wsum[threadIdx.x], wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (threadIdx.x >= (uint32_t)o) wi += u;
      }
      wsum[threadIdx.x] = wi - w;   // exclusive warp offsets
    }
    __syncthreads();
    const unsigned long long excl = carry + wsum[threadIdx.x >> 5] + incl - v;
    __syncthreads();
    if (i < nb) part[i] = excl;
    if (threadIdx.x == 1023) carry = excl + v;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) k_scan_write(const uint32_t* lw, uint64_t n,
                                                    const unsigned long long* part, uint64_t* offs) {
  __shared__ unsigned long long wsum[8];
  const uint64_t b0 = (uint64_t)blockIdx.x * kScanPerBlock;
  // each thread owns 16 consecutive lanes
  const uint64_t i0 = b0 + (uint64_t)threadIdx.x * 16;
  uint32_t v[16];
  unsigned long long s = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    v[k] = (i0 + k < n) ? lw[i0 + k] : 0u;
    s += v[k];
  }
  unsigned long long incl = s;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if ((threadIdx.x & 31) >= (uint32_t)o) incl += u;
  }
  if ((threadIdx.x & 31) == 31) wsum[threadIdx.x >> 5] = incl;
  __syncthreads();
  unsigned long long wbase = 0;
  for (uint32_t k = 0; k < (threadIdx.x >> 5); ++k) wbase += wsum[k];
  unsigned long long run = part[blockIdx.x] + wbase + incl - s;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t i = i0 + k;
    if (i < n) {
      offs[i] = 2ull * run;
      run += v[k];
      if (i + 1 == n) offs[n] = 2ull * run;
    }
  }
}

__global__ void __launch_bounds__(256) k_compact(const uint16_t* slots, const uint32_t* lw,
                                                 const uint64_t* offs, uint64_t n_lanes,
                                                 uint64_t slot_words, uint8_t* bs, uint64_t cap,
                                                 uint32_t* status) {
  const uint32_t lane = threadIdx.x & 31;
  const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
  for (uint64_t g = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < n_lanes; g += warps) {
    const uint32_t n = lw[g];
    const uint64_t dst = offs[g];
    if (dst + 2ull * n > cap) {
      if (lane == 0) atomicOr(status, SKV_FLAG_CAPACITY);
      continue;
    }
    const uint16_t* src = slots + (g + 1) * slot_words - n;
    uint16_t* d = reinterpret_cast<uint16_t*>(bs + dst);
    for (uint32_t k = lane; k < n; k += 32) d[k] = src[k];
  }
}

// Host-resident pipeline helpers: a group's lane offsets moved by a signed
// byte delta (decode: to the group's own stream), or by the running base of
// the joined stream (encode), which then advances past the group.
__global__ void k_offsets_shift(uint64_t* offs, uint64_t n, long long delta) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) offs[i] = (uint64_t)((long long)offs[i] + delta);
}
__global__ void k_offsets_rebase(uint64_t* offs, uint64_t n, const unsigned long long* base) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) offs[i] += *base;
}
__global__ void k_base_advance(unsigned long long* base, const uint64_t* offs_last) { *base = *offs_last; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SKV_OK : SKV_ERR_CUDA; }

int launch_check() { return cuda_status(cudaGetLastError()); }

template <typename Kern>
int set_smem(Kern k, int bytes) {
  return cuda_status(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
}

// blocks for a persistent codec kernel: one CTA per SM, warps spread so that
// every SM gets work when there are few chunks
void codec_grid(uint64_t n_chunks, int* blocks, int* threads, int max_threads) {
  int sms = sm_count();
  if (sms <= 0) sms = 1;
  uint64_t warps_per_block = (n_chunks + sms - 1) / sms;
  if (warps_per_block > (uint64_t)max_threads / 32) warps_per_block = max_threads / 32;
  if (warps_per_block < 1) warps_per_block = 1;
  uint64_t nb = (n_chunks + warps_per_block - 1) / warps_per_block;
  if (nb > (uint64_t)sms) nb = sms;
  if (nb * warps_per_block > kMaxWarps) nb = kMaxWarps / warps_per_block;
  *blocks = (int)(nb < 1 ? 1 : nb);
  *threads = (int)(warps_per_block * 32);
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* skv_status_string(int status) {
  switch (status) {
    case SKV_OK: return "ok";
    case SKV_ERR_INVALID_ARG: return "invalid argument";
    case SKV_ERR_CUDA: return "CUDA error";
    case SKV_ERR_CAPACITY: return "output buffer too small";
    case SKV_ERR_CORRUPT: return "corrupt bitstream";
    case SKV_ERR_TIMEOUT: return "timeout";
    case SKV_ERR_UNSUPPORTED: return "unsupported parameters";
    default: return "unknown status";
  }
}

int skv_check_params(const skv_params* p) {
  Geo g;
  return make_geo(p, &g);
}

uint64_t skv_num_positions(const skv_params* p) {
  Geo g;
  return make_geo(p, &g) == SKV_OK ? g.n_positions : 0;
}
uint64_t skv_num_channels(const skv_params* p) {
  Geo g;
  return make_geo(p, &g) == SKV_OK ? g.n_channels : 0;
}
uint32_t skv_num_tables(const skv_params* p) {
  Geo g;
  return make_geo(p, &g) == SKV_OK ? g.n_tables : 0;
}
uint64_t skv_num_chunks(const skv_params* p) {
  Geo g;
  return make_geo(p, &g) == SKV_OK ? g.n_chunks : 0;
}
uint64_t skv_num_lanes(const skv_params* p) {
  Geo g;
  return make_geo(p, &g) == SKV_OK ? g.n_lanes : 0;
}
uint64_t skv_tables_bytes(const skv_params* p) {
  Geo g;
  if (make_geo(p, &g) != SKV_OK) return 0;
  return (uint64_t)g.n_tables * (SKV_TABLE_STRIDE + (g.dtype == SKV_COEF_I16 ? SKV_TABLE_SLOT_BYTES : 0));
}
uint64_t skv_max_bitstream_bytes(const skv_params* p) {
  Geo g;
  if (make_geo(p, &g) != SKV_OK) return 0;
  return 4ull * g.n_lanes + 2ull * (1 + g.raw_bytes) * g.n_positions;
}
uint64_t skv_encode_workspace_bytes(const skv_params* p) {
  Geo g;
  if (make_geo(p, &g) != SKV_OK) return 0;
  return ws_layout(g).total;
}

static int calibrate_impl(const skv_params* p, const Paged* pg, uint32_t* d_status, const void* d_target,
                          const void* d_pred, uint8_t* d_bins, uint32_t* d_sum_abs, uint32_t* d_hist, void* stream) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pg && (st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s))) != SKV_OK) return st;
  if (g.n_channels == 0) return SKV_OK;
  if (!d_pred || !d_bins) return SKV_ERR_INVALID_ARG;
  if (g.dtype == SKV_COEF_I16) {
    if (d_sum_abs || d_hist) return SKV_ERR_INVALID_ARG;
    k_calibrate_coef<<<(unsigned)((g.C + 255) / 256), 256, 0, s>>>(static_cast<const float*>(d_pred), d_bins, g.C);
    return launch_check();
  }
  if (!d_target || !aligned16(d_target) || !aligned16(d_pred)) return SKV_ERR_INVALID_ARG;
  const uint32_t nc = (uint32_t)(p->n_calib < g.T ? p->n_calib : g.T);
  if (g.n_slices > 0x7FFFFFFFull) return SKV_ERR_UNSUPPORTED;
  const uint8_t* t8 = static_cast<const uint8_t*>(d_target);
  const uint8_t* p8 = static_cast<const uint8_t*>(d_pred);
  const Paged dense = {nullptr, 0, 0, 1};
  const unsigned nb = (unsigned)g.n_slices;
  if (g.esz == 1) {
    if (pg) k_calibrate_kv<1, true><<<nb, 256, 0, s>>>(t8, p8, d_bins, d_sum_abs, d_hist, g.T, g.D, nc, *pg, d_status, g.model);
    else k_calibrate_kv<1, false><<<nb, 256, 0, s>>>(t8, p8, d_bins, d_sum_abs, d_hist, g.T, g.D, nc, dense, nullptr, g.model);
  } else {
    if (pg) k_calibrate_kv<2, true><<<nb, 256, 0, s>>>(t8, p8, d_bins, d_sum_abs, d_hist, g.T, g.D, nc, *pg, d_status, 0u);
    else k_calibrate_kv<2, false><<<nb, 256, 0, s>>>(t8, p8, d_bins, d_sum_abs, d_hist, g.T, g.D, nc, dense, nullptr, 0u);
  }
  return launch_check();
}

int skv_calibrate(const skv_params* p, const void* d_target, const void* d_pred, uint8_t* d_bins,
                  uint32_t* d_sum_abs, uint32_t* d_hist, void* stream) {
  return calibrate_impl(p, nullptr, nullptr, d_target, d_pred, d_bins, d_sum_abs, d_hist, stream);
}

int skv_build_tables(const skv_params* p, void* d_tables, uint64_t tables_bytes, void* stream) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  if (!d_tables || !aligned16(d_tables) || tables_bytes < skv_tables_bytes(p)) return SKV_ERR_INVALID_ARG;
  k_build_tables<<<g.n_tables, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(d_tables), g.sub, g.dtype == SKV_COEF_I16 ? 1 : 0);
  return launch_check();
}

static int encode_impl(const skv_params* p, const Paged* pg, const void* d_target, const void* d_pred,
                       const void* d_tables, const uint8_t* d_bins, void* d_bitstream, uint64_t cap_bytes,
                       uint64_t* d_lane_offsets, void* d_workspace, uint64_t workspace_bytes, uint32_t* d_status,
                       uint64_t* h_total_bytes, void* stream) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!d_status || !d_lane_offsets || ((uintptr_t)d_status & 3) || ((uintptr_t)d_lane_offsets & 7))
    return SKV_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(g);
  if (g.n_lanes == 0) {
    st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
    if (st == SKV_OK) st = cuda_status(cudaMemsetAsync(d_lane_offsets, 0, 8, s));
    if (st == SKV_OK && h_total_bytes) {
      *h_total_bytes = 0;
      st = cuda_status(cudaStreamSynchronize(s));
    }
    return st;
  }
  if (!d_target || !d_pred || !d_tables || !d_bins || !d_bitstream || !d_workspace) return SKV_ERR_INVALID_ARG;
  if (!aligned16(d_target) || !aligned16(d_pred) || !aligned16(d_tables) || !aligned16(d_bins) ||
      !aligned16(d_workspace) || ((uintptr_t)d_bitstream & 1))
    return SKV_ERR_INVALID_ARG;
  if (workspace_bytes < wl.total) return SKV_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  CodecArgs a;
  memset(&a, 0, sizeof(a));
  a.k.k4096 = 4096u;
  a.k.minus1 = 0xFFFFFFFFu;
  a.k.k2p20 = 1u << 20;
  a.k.k8 = 8u;
  a.tgt = static_cast<const uint8_t*>(d_target);
  a.prd = static_cast<const uint8_t*>(d_pred);
  a.tables = static_cast<const uint8_t*>(d_tables);
  a.bins = d_bins;
  a.slots = reinterpret_cast<uint16_t*>(ws + wl.slots_off);
  a.lane_words = reinterpret_cast<uint32_t*>(ws + wl.lw_off);
  a.status = d_status;
  a.n_chunks = g.n_chunks;
  a.cps = g.cps;
  a.slice_pos = g.slice_pos;
  a.n_lanes = g.n_lanes;
  a.slot_words = g.slot_words;
  a.K = g.K;
  a.D = g.D;
  a.C = g.C;
  st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
  if (st != SKV_OK) return st;
  int blocks, threads;
  if (g.dtype != SKV_COEF_I16) {
    // one kernel: lanes coded into per-warp slots, chunks placed by look-back
    a.chunk_state = reinterpret_cast<unsigned long long*>(ws + wl.state_off);
    a.ticket = reinterpret_cast<unsigned long long*>(ws + wl.ticket_off);
    a.lane_offsets = d_lane_offsets;
    a.out_bs = static_cast<uint8_t*>(d_bitstream);
    a.cap = cap_bytes;
    a.slot_warps = wl.n_slots / (2 * kLanes);
    st = cuda_status(cudaMemsetAsync(ws + wl.state_off, 0, wl.total - wl.state_off, s));
    if (st != SKV_OK) return st;
    codec_grid(g.n_chunks, &blocks, &threads, kEncThreads);
    {
      uint64_t coding_warps = (uint64_t)blocks * (threads / 32);
      if (coding_warps > a.slot_warps) coding_warps = a.slot_warps;
      a.last_wave = g.n_chunks > coding_warps ? g.n_chunks - coding_warps : 0;
    }
    const int smem_bytes = (int)enc_smem_bytes((uint32_t)threads);
    const uint32_t smax = enc_smem_bytes(kEncThreads);
    if (pg) a.pg = *pg;
    auto run = [&](auto kern) -> int {
      int e = set_smem(kern, smax);
      if (e == SKV_OK) kern<<<blocks, threads, smem_bytes, s>>>(a);
      return e;
    };
    if (g.esz == 2) st = pg ? run(k_encode_kv<2, true, false>) : run(k_encode_kv<2, false, false>);
    else if (g.model) st = pg ? run(k_encode_kv<1, true, true>) : run(k_encode_kv<1, false, true>);
    else st = pg ? run(k_encode_kv<1, true, false>) : run(k_encode_kv<1, false, false>);
    if (st != SKV_OK) return st;
    if ((st = launch_check()) != SKV_OK) return st;
    if (h_total_bytes) {
      uint64_t total = 0;
      st = cuda_status(cudaMemcpyAsync(&total, d_lane_offsets + g.n_lanes, 8, cudaMemcpyDeviceToHost, s));
      if (st == SKV_OK) st = cuda_status(cudaStreamSynchronize(s));
      if (st != SKV_OK) return st;
      *h_total_bytes = total;
      if (total > cap_bytes) return SKV_ERR_CAPACITY;
    }
    return SKV_OK;
  }
  {
    // one warp per CTA: the few long lanes of a coefficient stream spread evenly over the SMs
    int sms = sm_count();
    const uint64_t cap_blocks = (uint64_t)(sms > 0 ? sms : 1) * 32;
    k_encode_coef<<<(unsigned)(g.n_chunks < cap_blocks ? g.n_chunks : cap_blocks), 32, 0, s>>>(a);
  }
  if ((st = launch_check()) != SKV_OK) return st;
  unsigned long long* part = reinterpret_cast<unsigned long long*>(ws + wl.part_off);
  k_scan_reduce<<<(unsigned)wl.n_scan_blocks, 256, 0, s>>>(a.lane_words, g.n_lanes, part);
  k_scan_parts<<<1, 1024, 0, s>>>(part, wl.n_scan_blocks);
  k_scan_write<<<(unsigned)wl.n_scan_blocks, 256, 0, s>>>(a.lane_words, g.n_lanes, part, d_lane_offsets);
  if ((st = launch_check()) != SKV_OK) return st;
  if (h_total_bytes) {
    uint64_t total = 0;
    st = cuda_status(cudaMemcpyAsync(&total, d_lane_offsets + g.n_lanes, 8, cudaMemcpyDeviceToHost, s));
    if (st == SKV_OK) st = cuda_status(cudaStreamSynchronize(s));
    if (st != SKV_OK) return st;
    *h_total_bytes = total;
    if (total > cap_bytes) return SKV_ERR_CAPACITY;
  }
  {
    int sms = sm_count();
    uint64_t nb = (g.n_lanes + 7) / 8;
    uint64_t cap_blocks = (uint64_t)(sms > 0 ? sms : 1) * 16;
    k_compact<<<(unsigned)(nb < cap_blocks ? nb : cap_blocks), 256, 0, s>>>(
        a.slots, a.lane_words, d_lane_offsets, g.n_lanes, g.slot_words, static_cast<uint8_t*>(d_bitstream),
        cap_bytes, d_status);
  }
  return launch_check();
}

static int decode_impl(const skv_params* p, const Paged* pg, const void* d_bitstream, uint64_t n_bytes,
                       const uint64_t* d_lane_offsets, const void* d_pred, const void* d_tables,
                       const uint8_t* d_bins, void* d_target_out, uint32_t* d_status, void* stream) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!d_status || ((uintptr_t)d_status & 3)) return SKV_ERR_INVALID_ARG;
  st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
  if (st != SKV_OK || g.n_lanes == 0) return st;
  if (!d_bitstream || !d_lane_offsets || !d_pred || !d_tables || !d_bins || !d_target_out)
    return SKV_ERR_INVALID_ARG;
  if (!aligned16(d_bitstream) || ((uintptr_t)d_lane_offsets & 7) || !aligned16(d_pred) ||
      !aligned16(d_tables) || !aligned16(d_bins) || !aligned16(d_target_out))
    return SKV_ERR_INVALID_ARG;
  CodecArgs a;
  memset(&a, 0, sizeof(a));
  a.prd = static_cast<const uint8_t*>(d_pred);
  a.out = static_cast<uint8_t*>(d_target_out);
  a.tables = static_cast<const uint8_t*>(d_tables);
  a.bins = d_bins;
  a.bs = static_cast<const uint8_t*>(d_bitstream);
  a.offs = d_lane_offsets;
  a.n_bytes = n_bytes;
  a.status = d_status;
  a.n_chunks = g.n_chunks;
  a.cps = g.cps;
  a.slice_pos = g.slice_pos;
  a.n_lanes = g.n_lanes;
  a.K = g.K;
  a.D = g.D;
  a.C = g.C;
  if (g.dtype == SKV_COEF_I16) {
    // one warp per CTA: the few long lanes of a coefficient stream spread evenly over the SMs
    int sms = sm_count();
    const uint64_t cap_blocks = (uint64_t)(sms > 0 ? sms : 1) * 32;
    k_decode_coef<<<(unsigned)(g.n_chunks < cap_blocks ? g.n_chunks : cap_blocks), 32, 0, s>>>(a);
    return launch_check();
  }
  int blocks, threads;
  const int max_threads = dec_threads(pg != nullptr, g.model != 0);
  codec_grid(g.n_chunks, &blocks, &threads, max_threads);
  const int smem_bytes = (int)(kDecTabBytes + (uint32_t)threads * kRingStride);
  const uint32_t smax = kDecTabBytes + max_threads * kRingStride;
  if (pg) a.pg = *pg;
  auto run = [&](auto kern) -> int {
    int e = set_smem(kern, smax);
    if (e == SKV_OK) kern<<<blocks, threads, smem_bytes, s>>>(a);
    return e;
  };
  if (g.esz == 2) st = pg ? run(k_decode_kv<2, true, false>) : run(k_decode_kv<2, false, false>);
  else if (g.model) st = pg ? run(k_decode_kv<1, true, true>) : run(k_decode_kv<1, false, true>);
  else st = pg ? run(k_decode_kv<1, true, false>) : run(k_decode_kv<1, false, false>);
  if (st != SKV_OK) return st;
  return launch_check();
}

int skv_encode(const skv_params* p, const void* d_target, const void* d_pred, const void* d_tables,
               const uint8_t* d_bins, void* d_bitstream, uint64_t cap_bytes, uint64_t* d_lane_offsets,
               void* d_workspace, uint64_t workspace_bytes, uint32_t* d_status, uint64_t* h_total_bytes,
               void* stream) {
  return encode_impl(p, nullptr, d_target, d_pred, d_tables, d_bins, d_bitstream, cap_bytes, d_lane_offsets,
                     d_workspace, workspace_bytes, d_status, h_total_bytes, stream);
}

int skv_decode(const skv_params* p, const void* d_bitstream, uint64_t n_bytes, const uint64_t* d_lane_offsets,
               const void* d_pred, const void* d_tables, const uint8_t* d_bins, void* d_target_out,
               uint32_t* d_status, void* stream) {
  return decode_impl(p, nullptr, d_bitstream, n_bytes, d_lane_offsets, d_pred, d_tables, d_bins, d_target_out,
                     d_status, stream);
}

// Paged pools: checks the layout against the parameters (host only).
static int paged_args(const skv_params* p, const skv_paged_layout* L, Paged* pg) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  if (g.dtype == SKV_COEF_I16) return SKV_ERR_UNSUPPORTED;
  if (!L || !L->d_block_table || ((uintptr_t)L->d_block_table & 3) || L->n_blocks == 0 || L->block_tokens == 0 ||
      (L->block_tokens & (L->block_tokens - 1)) != 0)
    return SKV_ERR_INVALID_ARG;
  uint32_t shift = 0;
  while ((1u << shift) < L->block_tokens) ++shift;
  pg->bt = L->d_block_table;
  pg->n_blocks = L->n_blocks;
  pg->shift = shift;
  pg->H = p->n_heads;
  return SKV_OK;
}

int skv_calibrate_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_target_pool,
                        const void* d_pred_pool, uint8_t* d_bins, uint32_t* d_sum_abs, uint32_t* d_hist,
                        uint32_t* d_status, void* stream) {
  Paged pg;
  int st = paged_args(p, layout, &pg);
  if (st != SKV_OK) return st;
  if (!d_status || ((uintptr_t)d_status & 3)) return SKV_ERR_INVALID_ARG;
  return calibrate_impl(p, &pg, d_status, d_target_pool, d_pred_pool, d_bins, d_sum_abs, d_hist, stream);
}

int skv_encode_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_target_pool,
                     const void* d_pred_pool, const void* d_tables, const uint8_t* d_bins, void* d_bitstream,
                     uint64_t cap_bytes, uint64_t* d_lane_offsets, void* d_workspace, uint64_t workspace_bytes,
                     uint32_t* d_status, uint64_t* h_total_bytes, void* stream) {
  Paged pg;
  int st = paged_args(p, layout, &pg);
  if (st != SKV_OK) return st;
  return encode_impl(p, &pg, d_target_pool, d_pred_pool, d_tables, d_bins, d_bitstream, cap_bytes, d_lane_offsets,
                     d_workspace, workspace_bytes, d_status, h_total_bytes, stream);
}

int skv_decode_paged(const skv_params* p, const skv_paged_layout* layout, const void* d_bitstream,
                     uint64_t n_bytes, const uint64_t* d_lane_offsets, const void* d_pred_pool,
                     const void* d_tables, const uint8_t* d_bins, void* d_target_pool_out, uint32_t* d_status,
                     void* stream) {
  Paged pg;
  int st = paged_args(p, layout, &pg);
  if (st != SKV_OK) return st;
  return decode_impl(p, &pg, d_bitstream, n_bytes, d_lane_offsets, d_pred_pool, d_tables, d_bins,
                     d_target_pool_out, d_status, stream);
}

uint64_t skv_ctx_scratch_bytes(uint64_t n_odd, uint32_t n_coef, uint32_t rank) {
  return align256(n_odd * n_coef * 2) + align256(n_odd * rank * 2) + 2 * align256((uint64_t)rank * n_coef * 2);
}

}  // extern "C"

namespace {
// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the driver library)
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}
// bf16 matrix [rows][inner] (row pitch inner * 2 bytes) read in 128-row x 64-column
// boxes in the 128-byte swizzle; out-of-range elements read as zero
int make_tmap(CUtensorMap* tm, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return SKV_ERR_UNSUPPORTED;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {kUmBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SKV_OK : SKV_ERR_INVALID_ARG;
}
}  // namespace

extern "C" {

int skv_ctx_means(const skv_ctx_map* map, const int16_t* d_q_even, uint64_t n_even, const float* d_mu_odd,
                  uint64_t n_odd, uint32_t n_coef, float* d_mu_out, void* d_scratch, uint64_t scratch_bytes,
                  uint32_t* d_status, void* stream) {
  if (!map || !map->d_V || !map->d_U || !d_status) return SKV_ERR_INVALID_ARG;
  const uint32_t R = map->rank, C = n_coef;
  if (R == 0 || R % 32 || R > 16384 || C == 0 || C % 32 || C > 16384 || map->shift1 > 30 || map->shift2 > 30)
    return SKV_ERR_INVALID_ARG;
  if (n_odd > n_even || n_odd > 65535ull * kUmBM) return SKV_ERR_INVALID_ARG;   // grid rows
  if (n_odd == 0) return SKV_OK;
  if (!d_q_even || !d_mu_odd || !d_mu_out || !d_scratch || !aligned16(d_q_even) || !aligned16(d_mu_odd) ||
      !aligned16(d_mu_out) || !aligned16(d_scratch) || !aligned16(map->d_V) || !aligned16(map->d_U))
    return SKV_ERR_INVALID_ARG;
  if (scratch_bytes < skv_ctx_scratch_bytes(n_odd, C, R)) return SKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* sp = static_cast<uint8_t*>(d_scratch);
  __nv_bfloat16* X = reinterpret_cast<__nv_bfloat16*>(sp);
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(sp + align256(n_odd * C * 2));
  __nv_bfloat16* Vb = reinterpret_cast<__nv_bfloat16*>(sp + align256(n_odd * C * 2) + align256(n_odd * R * 2));
  __nv_bfloat16* Ub = Vb + align256((uint64_t)R * C * 2) / 2;
  CUtensorMap tx, tv, tg, tu;
  int st = make_tmap(&tx, X, C, n_odd, kUmBM);
  if (st == SKV_OK) st = make_tmap(&tv, Vb, C, R, kUmBN);
  if (st == SKV_OK) st = make_tmap(&tg, G, R, n_odd, kUmBM);
  if (st == SKV_OK) st = make_tmap(&tu, Ub, R, C, kUmBN);
  if (st != SKV_OK) return st;
  // the attribute is per device: set on every call (a host-side call, no launch)
  if ((st = set_smem(k_ctx_umma<0>, (int)kUmSmem)) != SKV_OK || (st = set_smem(k_ctx_umma<1>, (int)kUmSmem)) != SKV_OK)
    return st;
  st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
  if (st != SKV_OK) return st;
  const uint64_t nw = (uint64_t)R * C;
  k_ctx_x<<<(unsigned)n_odd, 256, 0, s>>>(d_q_even, n_even, C, X);
  k_ctx_w<<<(unsigned)((nw + 255) / 256), 256, 0, s>>>(map->d_V, nw, Vb);
  k_ctx_w<<<(unsigned)((nw + 255) / 256), 256, 0, s>>>(map->d_U, nw, Ub);
  const unsigned gm = (unsigned)((n_odd + kUmBM - 1) / kUmBM);
  k_ctx_umma<0><<<dim3((R + kUmBN - 1) / kUmBN, gm), kUmThreads, kUmSmem, s>>>(tx, tv, (uint32_t)n_odd, R, C, map->shift1,
                                                                         G, nullptr, nullptr, d_status, 0u);
  k_ctx_umma<1><<<dim3((C + kUmBN - 1) / kUmBN, gm), kUmThreads, kUmSmem, s>>>(tg, tu, (uint32_t)n_odd, C, R, map->shift2,
                                                                         nullptr, d_mu_odd, d_mu_out, d_status, 0u);
  return launch_check();
}

int skv_selftest_ctx_wait(void* d_scratch, uint32_t* d_status, void* stream) {
  if (!d_scratch || !aligned16(d_scratch) || !d_status) return SKV_ERR_INVALID_ARG;
  // one 128 x 128 tile over a 128 x 64 bf16 operand in the scratch; no tile is ever loaded
  __nv_bfloat16* A = static_cast<__nv_bfloat16*>(d_scratch);
  __nv_bfloat16* G = A + kUmBM * kUmBK;
  CUtensorMap ta;
  int st = make_tmap(&ta, A, kUmBK, kUmBM, kUmBM);
  if (st != SKV_OK) return st;
  if ((st = set_smem(k_ctx_umma<0>, (int)kUmSmem)) != SKV_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
  if (st != SKV_OK) return st;
  k_ctx_umma<0><<<1, kUmThreads, kUmSmem, s>>>(ta, ta, kUmBM, kUmBN, kUmBK, 0, G, nullptr, nullptr, d_status, 1u);
  return launch_check();
}

// Scratch of skv_encode_noalloc: a file-scope device array, so the call never
// allocates.  Host code cannot use the symbol itself as a device address; the
// address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];
}  // namespace

int skv_encode_noalloc(const skv_params* p, const void* d_target, const void* d_pred, const void* d_tables,
                       const uint8_t* d_bins, void* d_bitstream, uint64_t cap_bytes, uint64_t* d_lane_offsets,
                       uint32_t* d_status, uint64_t* h_total_bytes, void* stream) {
  Geo g;
  int st = make_geo(p, &g);
  if (st != SKV_OK) return st;
  if (ws_layout(g).total > SKV_NOALLOC_SCRATCH_BYTES) return SKV_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SKV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SKV_ERR_CUDA;
      g_noalloc_ptr[dev] = ptr;
    }
    scratch = g_noalloc_ptr[dev];
  }
  return skv_encode(p, d_target, d_pred, d_tables, d_bins, d_bitstream, cap_bytes, d_lane_offsets, scratch,
                    SKV_NOALLOC_SCRATCH_BYTES, d_status, h_total_bytes, stream);
}

int skv_selftest_lookback(uint64_t* d_state, uint32_t n_chunks, uint32_t missing_chunk, uint32_t max_spins,
                          uint64_t* d_excl, uint32_t* d_status, void* stream) {
  if (!d_state || !d_excl || !d_status || n_chunks == 0 || n_chunks > 4096 || max_spins == 0)
    return SKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st = cuda_status(cudaMemsetAsync(d_state, 0, (size_t)n_chunks * 8, s));
  if (st == SKV_OK) st = cuda_status(cudaMemsetAsync(d_status, 0, 4, s));
  if (st == SKV_OK) st = cuda_status(cudaMemsetAsync(d_excl, 0xFF, (size_t)n_chunks * 8, s));
  if (st != SKV_OK) return st;
  const uint32_t warps_per_block = 8;
  k_selftest_lookback<<<(n_chunks + warps_per_block - 1) / warps_per_block, warps_per_block * 32, 0, s>>>(
      reinterpret_cast<unsigned long long*>(d_state), n_chunks, missing_chunk, max_spins, d_status,
      reinterpret_cast<unsigned long long*>(d_excl));
  return launch_check();
}

// ---------------------------------------------------------------------------
// Host-resident caches: layer groups coded on three streams (copy in, code,
// copy out), double-buffered device memory from the caller's workspace.
// ---------------------------------------------------------------------------
namespace {
struct HostPlan {
  Geo g;
  uint32_t group_layers, n_groups;
  uint64_t layer_elems, layer_lanes, layer_channels, group_cap;
  uint64_t in_bytes, off_bytes, ws_enc, total;
  uint64_t t_off[2], p_off[2], bs_off[2], o_off[2], ws_off, st_off, base_off;
};
int host_plan(const skv_params* p, uint32_t group_layers, uint64_t group_cap_bytes, HostPlan* hp) {
  memset(hp, 0, sizeof(*hp));
  int st = make_geo(p, &hp->g);
  if (st != SKV_OK) return st;
  if (hp->g.dtype == SKV_COEF_I16) return SKV_ERR_UNSUPPORTED;
  if (group_layers == 0 || p->n_layers == 0) return SKV_ERR_INVALID_ARG;
  const uint32_t gl = group_layers < p->n_layers ? group_layers : p->n_layers;
  hp->group_layers = gl;
  hp->n_groups = (p->n_layers + gl - 1) / gl;
  hp->layer_elems = (uint64_t)p->n_kv * p->n_heads * p->n_tokens * p->head_dim;
  hp->layer_lanes = hp->g.n_lanes / p->n_layers;
  hp->layer_channels = hp->g.n_channels / p->n_layers;
  skv_params q = *p;
  q.n_layers = gl;
  const uint64_t worst = skv_max_bitstream_bytes(&q);
  uint64_t cap = group_cap_bytes == 0 || group_cap_bytes > worst ? worst : group_cap_bytes;
  cap = (cap + 16 + 255) & ~255ull;   // + the decoder's read-ahead past the last byte
  hp->group_cap = cap;
  hp->in_bytes = align256(hp->layer_elems * gl * hp->g.esz);
  hp->off_bytes = align256((hp->layer_lanes * gl + 1) * 8);
  hp->ws_enc = align256(skv_encode_workspace_bytes(&q));
  uint64_t o = 0;
  for (int b = 0; b < 2; ++b) {
    hp->t_off[b] = o; o += hp->in_bytes;
    hp->p_off[b] = o; o += hp->in_bytes;
    hp->bs_off[b] = o; o += cap;
    hp->o_off[b] = o; o += hp->off_bytes;
  }
  hp->ws_off = o; o += hp->ws_enc;
  hp->st_off = o; o += align256(4ull * hp->n_groups);
  hp->base_off = o; o += 256;
  hp->total = o;
  return SKV_OK;
}
// combined status of n device words (synchronous)
int group_statuses(const uint32_t* d_st, uint32_t n, cudaStream_t s) {
  uint32_t buf[256];
  int worst = SKV_OK;
  for (uint32_t i = 0; i < n; i += 256) {
    const uint32_t m = n - i < 256 ? n - i : 256;
    int st = cuda_status(cudaMemcpyAsync(buf, d_st + i, 4 * m, cudaMemcpyDeviceToHost, s));
    if (st == SKV_OK) st = cuda_status(cudaStreamSynchronize(s));
    if (st != SKV_OK) return st;
    for (uint32_t k = 0; k < m; ++k) {
      const uint32_t v = buf[k];
      const int c = (v & SKV_FLAG_CORRUPT) ? SKV_ERR_CORRUPT : (v & SKV_FLAG_CAPACITY) ? SKV_ERR_CAPACITY
                    : (v & SKV_FLAG_TIMEOUT) ? SKV_ERR_TIMEOUT : (v & (SKV_FLAG_BAD_BIN | SKV_FLAG_BAD_BLOCK)) ? SKV_ERR_INVALID_ARG
                    : SKV_OK;
      if (worst == SKV_OK) worst = c;
    }
  }
  return worst;
}
struct Events {
  cudaEvent_t e[4][2];
  int n = 0;
  int create() {
    for (int i = 0; i < 4; ++i)
      for (int b = 0; b < 2; ++b) {
        if (cudaEventCreateWithFlags(&e[i][b], cudaEventDisableTiming) != cudaSuccess) return SKV_ERR_CUDA;
        ++n;
      }
    return SKV_OK;
  }
  ~Events() {
    for (int k = 0; k < n; ++k) cudaEventDestroy(e[k / 2][k % 2]);
  }
};
}  // namespace

uint64_t skv_host_workspace_bytes(const skv_params* p, uint32_t group_layers, uint64_t group_cap_bytes) {
  HostPlan hp;
  return host_plan(p, group_layers, group_cap_bytes, &hp) == SKV_OK ? hp.total : 0;
}

int skv_encode_host(const skv_params* p, const void* h_target, const void* h_pred, const void* d_tables,
                    uint8_t* d_bins, void* h_bitstream, uint64_t cap_bytes, uint64_t* h_lane_offsets,
                    uint64_t* h_total_bytes, uint32_t group_layers, uint64_t group_cap_bytes, void* d_workspace,
                    uint64_t workspace_bytes, void* const* streams) {
  HostPlan hp;
  int st = host_plan(p, group_layers, group_cap_bytes, &hp);
  if (st != SKV_OK) return st;
  if (!h_target || !h_pred || !d_tables || !d_bins || !h_bitstream || !h_lane_offsets || !d_workspace || !streams ||
      !aligned16(d_workspace) || !aligned16(d_tables) || !aligned16(d_bins) || workspace_bytes < hp.total)
    return SKV_ERR_INVALID_ARG;
  cudaStream_t s_in = static_cast<cudaStream_t>(streams[0]), s_c = static_cast<cudaStream_t>(streams[1]),
               s_out = static_cast<cudaStream_t>(streams[2]);
  Events ev;   // [0] inputs copied, [1] group coded, [2] offsets copied out, [3] stream copied out
  if ((st = ev.create()) != SKV_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  uint32_t* d_st = reinterpret_cast<uint32_t*>(ws + hp.st_off);
  unsigned long long* d_base = reinterpret_cast<unsigned long long*>(ws + hp.base_off);
  const uint32_t G = hp.n_groups, esz = hp.g.esz;
  const uint8_t* ht = static_cast<const uint8_t*>(h_target);
  const uint8_t* hpd = static_cast<const uint8_t*>(h_pred);
  uint8_t* hbs = static_cast<uint8_t*>(h_bitstream);
  if ((st = cuda_status(cudaMemsetAsync(d_base, 0, 8, s_c))) != SKV_OK) return st;
  if ((st = cuda_status(cudaMemsetAsync(d_st, 0, 4ull * G, s_c))) != SKV_OK) return st;
  auto lo_of = [&](uint32_t k) { return (uint64_t)k * hp.group_layers; };
  auto nl_of = [&](uint32_t k) {
    const uint64_t lo = lo_of(k);
    return (uint32_t)((lo + hp.group_layers <= p->n_layers ? hp.group_layers : p->n_layers - lo));
  };
  cudaEvent_t ev_first;
  if (cudaEventCreateWithFlags(&ev_first, cudaEventDisableTiming) != cudaSuccess) return SKV_ERR_CUDA;
  cudaEventRecord(ev_first, s_c);   // the memsets above come first on every stream
  cudaStreamWaitEvent(s_in, ev_first, 0);
  cudaStreamWaitEvent(s_out, ev_first, 0);
  auto copy_in = [&](uint32_t k) -> int {
    const uint32_t b = k & 1u;
    if (k >= 2 && cudaStreamWaitEvent(s_in, ev.e[1][b], 0) != cudaSuccess) return SKV_ERR_CUDA;
    const uint64_t n = hp.layer_elems * nl_of(k) * esz, off = hp.layer_elems * lo_of(k) * esz;
    if (cudaMemcpyAsync(ws + hp.t_off[b], ht + off, n, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(ws + hp.p_off[b], hpd + off, n, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaEventRecord(ev.e[0][b], s_in) != cudaSuccess)
      return SKV_ERR_CUDA;
    return SKV_OK;
  };
  // the group's stream out to the host at the base the device computed (the
  // host reads it from the group's copied offsets: one group behind)
  auto copy_stream_out = [&](uint32_t k) -> int {
    const uint32_t b = k & 1u;
    if (cudaEventSynchronize(ev.e[2][b]) != cudaSuccess) return SKV_ERR_CUDA;
    const uint64_t l0 = hp.layer_lanes * lo_of(k), nl = hp.layer_lanes * nl_of(k);
    const uint64_t a0 = h_lane_offsets[l0], a1 = h_lane_offsets[l0 + nl];
    if (a1 < a0 || a1 - a0 > hp.group_cap - 16) return SKV_ERR_CAPACITY;
    if (a1 > cap_bytes) return SKV_ERR_CAPACITY;
    if (cudaMemcpyAsync(hbs + a0, ws + hp.bs_off[b], a1 - a0, cudaMemcpyDeviceToHost, s_out) != cudaSuccess ||
        cudaEventRecord(ev.e[3][b], s_out) != cudaSuccess)
      return SKV_ERR_CUDA;
    return SKV_OK;
  };
  if ((st = copy_in(0)) != SKV_OK) goto done;
  for (uint32_t k = 0; k < G; ++k) {
    const uint32_t b = k & 1u;
    if (k + 1 < G && (st = copy_in(k + 1)) != SKV_OK) goto done;
    {
      skv_params q = *p;
      q.n_layers = nl_of(k);
      const uint64_t nlanes = hp.layer_lanes * q.n_layers;
      uint64_t* d_off = reinterpret_cast<uint64_t*>(ws + hp.o_off[b]);
      if (cudaStreamWaitEvent(s_c, ev.e[0][b], 0) != cudaSuccess ||
          (k >= 2 && cudaStreamWaitEvent(s_c, ev.e[3][b], 0) != cudaSuccess)) {
        st = SKV_ERR_CUDA;
        goto done;
      }
      uint8_t* bins_k = d_bins + hp.layer_channels * lo_of(k);
      if ((st = skv_calibrate(&q, ws + hp.t_off[b], ws + hp.p_off[b], bins_k, nullptr, nullptr, s_c)) != SKV_OK) goto done;
      if ((st = encode_impl(&q, nullptr, ws + hp.t_off[b], ws + hp.p_off[b], d_tables, bins_k, ws + hp.bs_off[b],
                            hp.group_cap - 16, d_off, ws + hp.ws_off, hp.ws_enc, d_st + k, nullptr, s_c)) != SKV_OK)
        goto done;
      const unsigned nb = (unsigned)((nlanes + 1 + 255) / 256);
      k_offsets_rebase<<<nb, 256, 0, s_c>>>(d_off, nlanes + 1, d_base);
      k_base_advance<<<1, 1, 0, s_c>>>(d_base, d_off + nlanes);
      if ((st = launch_check()) != SKV_OK || cudaEventRecord(ev.e[1][b], s_c) != cudaSuccess) {
        st = st != SKV_OK ? st : SKV_ERR_CUDA;
        goto done;
      }
      if (cudaStreamWaitEvent(s_out, ev.e[1][b], 0) != cudaSuccess ||
          cudaMemcpyAsync(h_lane_offsets + hp.layer_lanes * lo_of(k), d_off, 8 * (nlanes + 1), cudaMemcpyDeviceToHost,
                          s_out) != cudaSuccess ||
          cudaEventRecord(ev.e[2][b], s_out) != cudaSuccess) {
        st = SKV_ERR_CUDA;
        goto done;
      }
    }
    if (k >= 1 && (st = copy_stream_out(k - 1)) != SKV_OK) goto done;
  }
  st = copy_stream_out(G - 1);
done:
  {
    // drain all three streams before the events and buffers go away
    const int s1 = cuda_status(cudaStreamSynchronize(s_in)), s2 = cuda_status(cudaStreamSynchronize(s_c)),
              s3 = cuda_status(cudaStreamSynchronize(s_out));
    cudaEventDestroy(ev_first);
    if (st == SKV_OK) st = s1 != SKV_OK ? s1 : (s2 != SKV_OK ? s2 : s3);
  }
  if (st == SKV_OK) st = group_statuses(d_st, G, s_c);
  if (st == SKV_OK && h_total_bytes) *h_total_bytes = h_lane_offsets[hp.g.n_lanes];
  return st;
}

int skv_decode_host(const skv_params* p, const void* h_bitstream, uint64_t n_bytes, const uint64_t* h_lane_offsets,
                    const void* h_pred, const void* d_tables, const uint8_t* d_bins, void* h_target_out,
                    uint32_t group_layers, uint64_t group_cap_bytes, void* d_workspace, uint64_t workspace_bytes,
                    void* const* streams) {
  HostPlan hp;
  int st = host_plan(p, group_layers, group_cap_bytes, &hp);
  if (st != SKV_OK) return st;
  if (!h_bitstream || !h_lane_offsets || !h_pred || !d_tables || !d_bins || !h_target_out || !d_workspace ||
      !streams || !aligned16(d_workspace) || !aligned16(d_tables) || !aligned16(d_bins) ||
      workspace_bytes < hp.total)
    return SKV_ERR_INVALID_ARG;
  if (h_lane_offsets[0] != 0 || h_lane_offsets[hp.g.n_lanes] != n_bytes) return SKV_ERR_CORRUPT;
  cudaStream_t s_in = static_cast<cudaStream_t>(streams[0]), s_c = static_cast<cudaStream_t>(streams[1]),
               s_out = static_cast<cudaStream_t>(streams[2]);
  Events ev;   // [0] inputs copied, [1] group decoded, [2] target copied out
  if ((st = ev.create()) != SKV_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  uint32_t* d_st = reinterpret_cast<uint32_t*>(ws + hp.st_off);
  const uint32_t G = hp.n_groups, esz = hp.g.esz;
  const uint8_t* hbs = static_cast<const uint8_t*>(h_bitstream);
  const uint8_t* hpd = static_cast<const uint8_t*>(h_pred);
  uint8_t* hto = static_cast<uint8_t*>(h_target_out);
  auto lo_of = [&](uint32_t k) { return (uint64_t)k * hp.group_layers; };
  auto nl_of = [&](uint32_t k) {
    const uint64_t lo = lo_of(k);
    return (uint32_t)((lo + hp.group_layers <= p->n_layers ? hp.group_layers : p->n_layers - lo));
  };
  // every group's stream must fit its buffer (checked before anything is launched)
  for (uint32_t k = 0; k < G; ++k) {
    const uint64_t l0 = hp.layer_lanes * lo_of(k), nl = hp.layer_lanes * nl_of(k);
    const uint64_t a0 = h_lane_offsets[l0], a1 = h_lane_offsets[l0 + nl];
    if (a1 < a0 || a1 > n_bytes) return SKV_ERR_CORRUPT;
    if (a1 - a0 > hp.group_cap - 16) return SKV_ERR_CAPACITY;
  }
  for (uint32_t k = 0; k < G; ++k) {
    const uint32_t b = k & 1u;
    skv_params q = *p;
    q.n_layers = nl_of(k);
    const uint64_t l0 = hp.layer_lanes * lo_of(k), nlanes = hp.layer_lanes * q.n_layers;
    const uint64_t a0 = h_lane_offsets[l0], a1 = h_lane_offsets[l0 + nlanes];
    const uint64_t n = hp.layer_elems * q.n_layers * esz, off = hp.layer_elems * lo_of(k) * esz;
    uint64_t* d_off = reinterpret_cast<uint64_t*>(ws + hp.o_off[b]);
    // in: prediction, the group's stream and its offsets (moved to the group's own stream)
    if ((k >= 2 && cudaStreamWaitEvent(s_in, ev.e[1][b], 0) != cudaSuccess) ||
        cudaMemcpyAsync(ws + hp.p_off[b], hpd + off, n, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(ws + hp.bs_off[b], hbs + a0, a1 - a0, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaMemcpyAsync(d_off, h_lane_offsets + l0, 8 * (nlanes + 1), cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
        cudaEventRecord(ev.e[0][b], s_in) != cudaSuccess) {
      st = SKV_ERR_CUDA;
      break;
    }
    if (cudaStreamWaitEvent(s_c, ev.e[0][b], 0) != cudaSuccess ||
        (k >= 2 && cudaStreamWaitEvent(s_c, ev.e[2][b], 0) != cudaSuccess)) {
      st = SKV_ERR_CUDA;
      break;
    }
    k_offsets_shift<<<(unsigned)((nlanes + 1 + 255) / 256), 256, 0, s_c>>>(d_off, nlanes + 1, -(long long)a0);
    if ((st = launch_check()) != SKV_OK) break;
    if ((st = decode_impl(&q, nullptr, ws + hp.bs_off[b], a1 - a0, d_off, ws + hp.p_off[b], d_tables,
                          d_bins + hp.layer_channels * lo_of(k), ws + hp.t_off[b], d_st + k, s_c)) != SKV_OK)
      break;
    if (cudaEventRecord(ev.e[1][b], s_c) != cudaSuccess || cudaStreamWaitEvent(s_out, ev.e[1][b], 0) != cudaSuccess ||
        cudaMemcpyAsync(hto + off, ws + hp.t_off[b], n, cudaMemcpyDeviceToHost, s_out) != cudaSuccess ||
        cudaEventRecord(ev.e[2][b], s_out) != cudaSuccess) {
      st = SKV_ERR_CUDA;
      break;
    }
  }
  const int s1 = cuda_status(cudaStreamSynchronize(s_in)), s2 = cuda_status(cudaStreamSynchronize(s_c)),
            s3 = cuda_status(cudaStreamSynchronize(s_out));
  if (st == SKV_OK) st = s1 != SKV_OK ? s1 : (s2 != SKV_OK ? s2 : s3);
  if (st == SKV_OK) st = group_statuses(d_st, G, s_c);
  return st;
}

int skv_checked_failures(uint32_t* h_count, uint32_t* h_first_site) {
#if SKV_CHECKED
  if (!h_count || !h_first_site) return SKV_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return SKV_ERR_CUDA;
  if (cudaMemcpyFromSymbol(h_count, g_check_count, 4) != cudaSuccess ||
      cudaMemcpyFromSymbol(h_first_site, g_check_site, 4) != cudaSuccess)
    return SKV_ERR_CUDA;
  const uint32_t z = 0;
  if (cudaMemcpyToSymbol(g_check_count, &z, 4) != cudaSuccess || cudaMemcpyToSymbol(g_check_site, &z, 4) != cudaSuccess)
    return SKV_ERR_CUDA;
  return SKV_OK;
#else
  (void)h_count;
  (void)h_first_site;
  return SKV_ERR_UNSUPPORTED;
#endif
}

int skv_read_status(const uint32_t* d_status, void* stream) {
  if (!d_status) return SKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  int st = cuda_status(cudaMemcpyAsync(&v, d_status, 4, cudaMemcpyDeviceToHost, s));
  if (st == SKV_OK) st = cuda_status(cudaStreamSynchronize(s));
  if (st != SKV_OK) return st;
  if (v & SKV_FLAG_CORRUPT) return SKV_ERR_CORRUPT;
  if (v & SKV_FLAG_CAPACITY) return SKV_ERR_CAPACITY;
  if (v & SKV_FLAG_TIMEOUT) return SKV_ERR_TIMEOUT;
  if (v & (SKV_FLAG_BAD_BIN | SKV_FLAG_BAD_BLOCK)) return SKV_ERR_INVALID_ARG;
  return SKV_OK;
}

}  // extern "C"
