// The two expert GEMMs of the W4A16 fused MoE feed-forward on the 5th-generation
// tensor cores (tcgen05), one persistent warp-specialised kernel template:
//
//   gate/up:  [g; u] = W1[e] . x_t   (W1 rows interleaved gate/up), epilogue
//             h = SiLU(g) * u -> fp16 intermediate (blocked layout)
//   down:     y = W2[e] . h_r,  epilogue acc[t] += topk_weight * y  (fp32 red.add)
//
// Tensor-core operands are fp16 (kind::f16, fp32 accumulate): the dequantised
// weights are exact in fp16, and the bf16 hidden states convert to fp16 exactly
// inside fp16's range (the gather saturates beyond +-65504).
//
// "Swap-AB" orientation: the 128 weight rows of a tile are the MMA M dimension
// and the routed tokens of one expert (16..64, a multiple of 16) are MMA N, so a
// single token (decode) costs one N=16 tile instead of a 128-row tile.
//
// The pipeline moves in steps of 128 reduction elements (two 64-element k-blocks
// of the packed layout): every per-step cost (barrier tests and arrivals, MMA
// commits, copy issue, address arithmetic) is paid once per 128 elements.
//
// Per CTA (one per SM), 24 warps:
//   warp 0       one lane bulk-copies the packed INT4 weights, 2 steps (18 KB) per
//                copy, into a 4-chunk ring
//   warp 1       4 lanes bulk-copy the activation tile (B operand, both 64-element
//                planes of a step) into an 8-step ring of its own (the lanes issue
//                4 consecutive steps at once); running the small, L2-resident
//                copies that far ahead takes their latency off the MMA path
//   warps 2, 3   tcgen05.mma issuers for alternate steps (8 MMAs each), each into
//                its own accumulators (warp 2 also allocates tensor memory)
//   warps 4..19  dequantise INT4 -> fp16 in registers and store the A operand
//                straight into tensor memory (tcgen05.st) through a 4-stage ring;
//                four warps per lane quadrant, warp `phase` converting the steps
//                phase, phase + 4, ... and so always writing stage `phase`
//   warps 20..23 epilogue: tcgen05.ld of both issuers' fp32 accumulators
//                (double-buffered), summed
//
// The dequantisation writes the weight tile into tensor memory rather than
// shared memory, so shared-memory bandwidth carries only the packed codes and the
// activations; the MMA reads A from tensor memory and B from shared memory.
//
// Work split (stream-K): the units (expert, 128-row weight tile, token tile) each
// have KBn steps of 128 reduction elements; all units' steps are laid end to end
// and every CTA takes an equal contiguous share. Every SM therefore streams the
// same number of weight bytes whatever the routing. A unit cut between CTAs is
// finished by its last contributor: down-GEMM partials are simply added into the
// fp32 accumulator; gate/up partials go to a per-CTA scratch slot, and the CTA
// whose atomic ticket completes the unit's step count sums the slots in CTA
// order (deterministic), applies SiLU*up and writes the tile. No CTA ever waits
// for another.
//
// Warp-collective tcgen05 instructions (.sync.aligned: st, ld, wait, alloc,
// dealloc) are always preceded by a warp-wide synchronisation, never issued right
// after lane-divergent code.
//
// Every mbarrier wait is bounded in time (see mbar_wait); a wait that gives up
// raises a CTA-wide abort flag, records MOE_W4A16_STATUS_TIMEOUT, and all roles
// fall through to the teardown, which still waits for in-flight copies and MMAs
// and frees tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "rowcopy.cuh"
#include "small_route.cuh"
#include "stream_k.cuh"

namespace moe {

// Optional pipeline timeline for performance work: built with -DMOE_GEMM_TRACE,
// CTA 0 of the traced GEMM records clock64() at fixed points per step into a
// device array read back with moe_gemm_trace_read(). Compiled out otherwise.
#ifdef MOE_GEMM_TRACE
__device__ long long g_gemm_trace[16][2048];
extern "C" int moe_gemm_trace_read(long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_gemm_trace, sizeof(g_gemm_trace)));
}
extern "C" int moe_gemm_wait_iters(unsigned long long* host, int reset) {
  int e = static_cast<int>(cudaMemcpyFromSymbol(host, g_wait_iters, sizeof(g_wait_iters)));
  if (reset) {
    unsigned long long z[32] = {};
    cudaMemcpyToSymbol(g_wait_iters, z, sizeof(z));
  }
  return e;
}
#ifndef MOE_GEMM_TRACE_MODE
#define MOE_GEMM_TRACE_MODE 1
#endif
#define TRACE_POINT(slot, idx)                                                      \
  do {                                                                              \
    if (blockIdx.x == 0 && kMode == MOE_GEMM_TRACE_MODE && (idx) < 2048)            \
      g_gemm_trace[(slot)][(idx)] = clock64();                                      \
  } while (0)
// every CTA of both GEMMs: global-timer stamps of a few events (latest wins)
__device__ unsigned long long g_cta_trace[3][256][16];
extern "C" int moe_gemm_cta_trace_read(unsigned long long* host, int reset) {
  int e = static_cast<int>(cudaMemcpyFromSymbol(host, g_cta_trace, sizeof(g_cta_trace)));
  if (reset) {
    static unsigned long long z[3 * 256 * 16];
    cudaMemcpyToSymbol(g_cta_trace, z, sizeof(z));
  }
  return e;
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define CTA_STAMP(ev)                                                               \
  do {                                                                              \
    if (blockIdx.x < 256) atomicMax(&g_cta_trace[kMode - 1][blockIdx.x][(ev)], gtimer()); \
  } while (0)
#else
#define CTA_STAMP(ev) \
  do {                \
  } while (0)
#define TRACE_POINT(slot, idx) \
  do {                         \
  } while (0)
#endif

namespace {

// Dequantisation warps per TMEM lane quadrant (compile-time; 4 by default, one
// per operand stage).
#ifndef MOE_DEQ_PHASES
#define MOE_DEQ_PHASES 4
#endif
constexpr int kDeqPhases = MOE_DEQ_PHASES;
constexpr int kWarpW = 0, kWarpB = 1, kWarpMma0 = 2, kWarpMma1 = 3, kWarpDeq0 = 4;
constexpr int kWarpEpi0 = kWarpDeq0 + 4 * kDeqPhases;
constexpr int kThreads = (kWarpEpi0 + 4) * 32;
// A pipeline step covers kSub consecutive 64-element k-blocks (128 reduction
// elements): every per-step cost (barrier waits and arrivals, MMA commit, address
// arithmetic) is paid once per 128 elements.
constexpr int kSub = 2;
constexpr int kWStepBytes = kSub * kWBlockBytes;  // packed weights of one step (9 KB)
constexpr int kWChunk = 2;               // steps per weight copy (one 18 KB bulk copy)
constexpr int kWChunkBytes = kWChunk * kWStepBytes;
// A operand stage ring in tensor memory: 6 stages when the CTA's widest token tile
// has at most two row groups (the accumulators then take at most 4 x 32 columns),
// else 4. More stages give each dequantisation warp more slack between storing a
// stage and needing it again.
constexpr int kNS = 4;                   // stages with tiles of three or four row groups
constexpr int kNSNarrow = 4;             // stages with tiles of at most two row groups
constexpr int kNSMax = kNSNarrow;
constexpr int kTmemCols = 512;
constexpr int kACols = kSub * 32;        // one step of fp16 A: 128 lanes x 64 columns
// accumulators follow the A ring: 4 of them (2 issuers x 2 buffers), each as wide
// as the CTA's widest token tile
constexpr int kProducerLanes = 4;        // copy-issuing threads per producer warp

// The two shared-memory rings (packed weights, activation tiles) divide one
// region between them per CTA: a B stage holds a step of the CTA's widest token
// tile (16..64 rows), and the rings are as deep as that allows. Both rings hold
// the same number of steps: the bulk-copy engine serves an SM's copies in issue
// order, so an activation copy issued behind a long run of weight copies lands
// late and stalls the MMA. With equal depths the B copy of a step is issued just
// after the weight copy of the same step (its slot frees with the MMA that
// follows the conversion which frees the weight slot) and lands with it.
constexpr int kMaxNWS = 8;               // weight ring depth limit in chunks
constexpr int kMaxNB = 2 * kMaxNWS;      // B ring depth limit in steps
constexpr int kBRowGroupStep = kSub * kRowGroupBytes;  // B bytes of one row group per step
// barrier indices
constexpr int kBarWFull = 0;                     // weight chunk landed (bulk-copy bytes)
constexpr int kBarWEmpty = kBarWFull + kMaxNWS;  // weight chunk read (4 dequant warps per step)
constexpr int kBarFull = kBarWEmpty + kMaxNWS;   // A stage ready: stored by its 4 dequant warps
constexpr int kBarEmpty = kBarFull + kNSMax;     // A stage consumed by the MMAs (tcgen05.commit)
constexpr int kBarBFull = kBarEmpty + kNSMax;    // B stage landed (bulk-copy bytes)
constexpr int kBarBEmpty = kBarBFull + kMaxNB;   // B stage consumed by the MMAs (tcgen05.commit)
constexpr int kBarAccFull = kBarBEmpty + kMaxNB; // [issuer][buffer]: accumulator complete
constexpr int kBarAccEmpty = kBarAccFull + 4;    // [buffer]: epilogue has read both issuers' sums
constexpr int kBarDrain = kBarAccEmpty + 2;      // [issuer]
constexpr int kBarNever = kBarDrain + 2;         // nothing ever arrives (the give-up test hook)
constexpr int kNumBars = kBarNever + 1;
// fixed part of shared memory first, then the ring region
constexpr int kSmStage = 0;                              // SwiGLU staging tile (1024-aligned)
constexpr int kSmBar = kSmStage + kBNMax * 128;
constexpr int kSmMisc = kSmBar + kNumBars * 8;
constexpr int kMaxSegs = 256;            // units decoded into shared memory up front
constexpr int kSmSeg = kSmMisc + 64;
constexpr int kSmSched = kSmSeg + kMaxSegs * 16;  // [kMaxCtas + 1] stream-K boundaries
constexpr int kSmSmall = kSmSched + (kMaxCtas + 1) * 8 + 8;  // [kSmallTiles] TokenTile + count
constexpr int kSmRings = ((kSmSmall + kSmallTiles * 16 + 16 + 1023) / 1024) * 1024;
constexpr int kSmAlloc = 227 * 1024;     // the whole per-CTA limit (base aligned to 1024 inside)
constexpr int kRingBytes = kSmAlloc - 1024 - kSmRings;
static_assert(kSmRings < kSmAlloc - 1024, "shared memory budget");
static_assert(2 * kSmallPadRows * 4 <= kMaxSegs * 16,
              "the fused launch's padded row list takes the segment table's place");
static_assert(kNS * kACols + 4 * kBNMax <= kTmemCols && kNSNarrow * kACols + 4 * 32 <= kTmemCols,
              "tensor memory budget");
static_assert(kWChunk == 2, "the chunk arithmetic below assumes 2-step chunks");

// Ring depths for a CTA whose widest token tile has `ng` row groups: nws weight
// chunks (an even number: the parity arguments below need even depths) and
// nb = 2 * nws B stages of ng row groups -- 8 chunks / 16 steps for one-group
// tiles, 6 / 12 for two, 4 / 8 for three or four.
struct RingCfg {
  int nb, nws;
  uint32_t b_stage, b_plane;  // bytes of one B stage, and of one 64-element plane in it
};
__host__ __device__ constexpr RingCfg ring_cfg(int ng) {
  const int g = ng < 1 ? 1 : (ng > kBNMax / kRowGroup ? kBNMax / kRowGroup : ng);
  const int b_stage = g * kBRowGroupStep;
  int nws = kRingBytes / (kWChunkBytes + 2 * b_stage);
  nws = nws > kMaxNWS ? kMaxNWS : nws;
  nws &= ~1;
  return RingCfg{2 * nws, nws, static_cast<uint32_t>(b_stage), static_cast<uint32_t>(g * kRowGroupBytes)};
}
static_assert(ring_cfg(1).nws == 8 && ring_cfg(2).nws == 6 && ring_cfg(3).nws == 4 &&
                  ring_cfg(4).nws == 4,
              "ring depths as documented");
static_assert(ring_cfg(1).nb * ring_cfg(1).b_stage + ring_cfg(1).nws * kWChunkBytes <= kRingBytes &&
                  ring_cfg(2).nb * ring_cfg(2).b_stage + ring_cfg(2).nws * kWChunkBytes <= kRingBytes &&
                  ring_cfg(4).nb * ring_cfg(4).b_stage + ring_cfg(4).nws * kWChunkBytes <= kRingBytes,
              "rings fit the region");

// Stage-reuse safety. A dequantisation warp reuses A stage st for step it after
// a parity test of Empty[st], meaning "the MMA of step it - kNS is done". A
// parity test cannot tell that phase from the one two uses back, so the warp must
// already know that the MMA of it - 2*kNS has completed, or it may overwrite the
// stage under a running MMA and arrive in the wrong phase of Full[st]. It knows
// this from its own earlier waits: j iterations back it waited for the MMA of
// it - j*kDeqPhases - kNS, and each issuer (issuers alternate by step parity)
// completes its steps in order, so that wait covers it - 2*kNS whenever
// j*kDeqPhases <= kNS and j*kDeqPhases - kNS is even.
constexpr bool stage_reuse_is_safe(int phases, int stages) {
  for (int j = 1; j * phases <= stages; ++j)
    if ((stages - j * phases) % 2 == 0) return true;
  return false;
}
static_assert(stage_reuse_is_safe(kDeqPhases, kNS) && stage_reuse_is_safe(kDeqPhases, kNSNarrow),
              "a dequantisation warp could pass a stale Empty phase (parity aliasing)");
// The MMA issuer that waits on a B (or A) stage for step it consumed the
// previous phase itself (step it - depth) only if the depth is even; a B
// producer lane reuses a slot only after an earlier lockstep iteration. A
// dequantisation warp sees every second weight chunk (its steps are 4 apart, 2
// steps a chunk), so with an even weight ring it has itself waited for the
// previous phase of every chunk slot it waits on.
static_assert(kMaxNB % 2 == 0 && kNS % 2 == 0 && kNSNarrow % 2 == 0 &&
                  kNS >= kDeqPhases && kNSNarrow >= kDeqPhases && ring_cfg(4).nb >= kProducerLanes &&
                  kDeqPhases == 2 * kWChunk,
              "ring depths must be even and the B ring at least as deep as the producer lanes");

constexpr int kEpiWarps = 4, kEpiThreads = 128;
constexpr int kEpiBar = 1;  // named barrier id of the epilogue warps
constexpr int kRowRegs = kBNMax / 32;  // token rows per epilogue lane (routing prefetch)

struct Unit {
  int e, rt, g0, ng;
};

// Units are ordered [expert][row tile][token tile of that expert], so the token
// tiles sharing one weight tile run back to back (the re-read hits L2).
__device__ __forceinline__ Unit decode_unit(long long u, int R, const TokenTile* tiles,
                                            const int32_t* expert_tiles) {
  const TokenTile a = tiles[u / R];
  const int te = expert_tiles[a.expert];
  const long long up = u - static_cast<long long>(R) * a.first;
  Unit r;
  r.e = a.expert;
  r.rt = static_cast<int>(up / te);
  const TokenTile b = tiles[a.first + static_cast<int>(up % te)];
  r.g0 = b.g0;
  r.ng = b.ngroups;
  return r;
}

// The units of this CTA's share, decoded once at kernel start into shared memory
// (consecutive segments are consecutive units): the roles then never stall at a
// unit boundary on the dependent global loads of decode_unit. Units beyond the
// table are decoded on the fly.
static_assert(sizeof(Unit) == 16, "segment table entry size");
// A batch of at most 32 routed slots has at most one token tile per expert, so
// unit u is (tile u / R, row tile u % R); its tiles live in shared memory.
__device__ __forceinline__ Unit decode_unit_small(long long u, int R, const TokenTile* tiles) {
  const TokenTile a = tiles[u / R];
  Unit r;
  r.e = a.expert;
  r.rt = static_cast<int>(u % R);
  r.g0 = a.g0;
  r.ng = a.ngroups;
  return r;
}

struct SegTable {
  const Unit* t;
  long long u0;
  int n, R;
  const TokenTile* tiles;
  const int32_t* expert_tiles;
  const TokenTile* small_tiles;  // the small-batch tile list (shared memory), or null
  __device__ __forceinline__ Unit get(long long u) const {
    const long long s = u - u0;
    if (s >= 0 && s < n) return t[s];
    return small_tiles ? decode_unit_small(u, R, small_tiles) : decode_unit(u, R, tiles, expert_tiles);
  }
};

// Random access into this CTA's step sequence for lanes that walk through it
// together: seek(it) moves forward to the segment holding sequence index `it`.
struct Cursor {
  SegIter si;
  long long u = 0, seg_it0 = 0;
  int kb0 = 0, kb1 = 0;
  bool valid = false, decoded = false;
  Unit un{};
  SegTable segs;
  __device__ Cursor(long long begin, long long end, int KBn, const SegTable& st)
      : si(begin, end, KBn), segs(st) {
    valid = si.next(u, kb0, kb1);
  }
  __device__ __forceinline__ bool seek(long long it, int& kb) {
    while (valid && it >= seg_it0 + (kb1 - kb0)) {
      seg_it0 += kb1 - kb0;
      valid = si.next(u, kb0, kb1);
      decoded = false;
    }
    if (!valid) return false;
    if (!decoded) {
      un = segs.get(u);
      decoded = true;
    }
    kb = kb0 + static_cast<int>(it - seg_it0);
    return true;
  }
};

// 32 INT4 codes (one scale group) -> 16 f16x2 words, columns of the A operand.
// The repack places each pair of codes (u_lo, u_hi) of a word at bits 6..9 and
// 22..25 (directly, after a shift left or right by 4, or after a rotation by 8):
// OR-ing them below the exponent of fp16 16.0 gives the pair 16 + u exactly, and
// one fused multiply-add with the scale s and -24 s gives (16 + u) s - 24 s =
// (u - 8) s, rounded once. It is exact: -24 s = -3 * 8 s has at most 10
// significant bits for a bf16 scale (8), and (u - 8) s at most 3 + 8, so both are
// fp16 numbers for scales in [2^-14, 2720] (the repack rejects others). Per word
// of eight codes: 3 shifts, 4 three-input logic ops, 4 fma. `s2` is the fp16 scale
// in both halves.
__device__ __forceinline__ uint32_t or_masked(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;  // (a & mask) | bits in one three-input logic op
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}
__device__ __forceinline__ void dequant_group(const uint4 qv, const uint32_t s2, uint32_t* out) {
  const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
  const uint32_t c2 = f16x2_mul(s2, 0xCE00CE00u);  // -24 s in both halves (exact)
  constexpr uint32_t kMask = 0x03C003C0u, kSixteen = 0x4C004C00u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t q = w[j];
    out[4 * j + 0] = f16x2_fma(or_masked(q, kMask, kSixteen), s2, c2);        // codes 0, 1
    out[4 * j + 1] = f16x2_fma(or_masked(q << 4, kMask, kSixteen), s2, c2);   // codes 2, 3
    out[4 * j + 2] = f16x2_fma(or_masked(q >> 4, kMask, kSixteen), s2, c2);   // codes 4, 5
    out[4 * j + 3] = f16x2_fma(or_masked(__funnelshift_l(q, q, 8), kMask, kSixteen), s2, c2);  // 6, 7
  }
}

// fp16 bits of x, saturated to the finite range (+-65504).
__device__ __forceinline__ uint16_t f16_bits_sat(float x) {
  x = fminf(fmaxf(x, -65504.0f), 65504.0f);
  return __half_as_ushort(__float2half_rn(x));
}

// SiLU(gate) * up for one 16-column chunk of the accumulator and store into the
// staging tile (blocked, swizzled). Lanes (2i, 2i+1) hold the gate and up rows of
// feature i for the chunk's 16 tokens; the even lane finishes tokens 0..7 and the
// odd lane tokens 8..15, so each sends its partner the half the partner finishes.
// No lane-divergent code: every lane evaluates 8 SiLUs. The sigmoid uses the fast
// reciprocal (a few fp32 ulps, far below the fp16 rounding of h; it tends to 0 as
// e^-g overflows to infinity).
// Token row R of the tile was fed in as x * 2^-e (e = the row's prescale
// exponent, held by lane R % 32 in e_reg, the register of R / 32): the sums are
// multiplied back by 2^e before SiLU, and h is stored as h * 2^-2e (the down
// GEMM's epilogue multiplies by 2^2e). A padding row (exponent kPadRowExp) has no
// operand data: its h is stored as zero. Returns true if a stored value had to be
// saturated to fp16's range.
__device__ __forceinline__ bool swiglu_chunk(const float (&v)[16], int chunk, int quad, int lane,
                                             uint32_t s_stage, int e_reg) {
  const bool is_gate = (lane & 1) == 0;
  const int f = quad * 16 + (lane >> 1);
  const int row0 = chunk * 16 + (is_gate ? 0 : 8);
  bool sat = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float mine = is_gate ? v[j] : v[j + 8];
    const float other = __shfl_xor_sync(0xffffffffu, is_gate ? v[j + 8] : v[j], 1);
    const int e_raw = __shfl_sync(0xffffffffu, e_reg, (row0 + j) & 31);
    const bool pad = e_raw == kPadRowExp;
    const int e = pad ? 0 : (e_raw < -kMaxRowExp ? -kMaxRowExp : (e_raw > kMaxRowExp ? kMaxRowExp : e_raw));
    const float up_scale = exp2_int(e);
    const float g = (is_gate ? mine : other) * up_scale;
    const float u = (is_gate ? other : mine) * up_scale;
    const float sig = __fdividef(1.0f, 1.0f + __expf(-g));
    const float h = pad ? 0.0f : g * sig * u * exp2_int(-2 * e);
    sat = sat || fabsf(h) > 65504.0f;
    st_shared_u16(s_stage + blocked_offset(row0 + j, f), f16_bits_sat(h));
  }
  return sat;
}

// The fused launch's preparation, by the 128 epilogue threads of every CTA before
// their first segment: CTA c takes padded rows c, c + G, ...: records the row's
// slot, and for a real row its prescale exponent and its copy as scaled fp16 in
// the blocked B layout (the expert's packing order under act-order), as the
// routing + gather kernel does for the separate launches; then zeroes its slice of
// the output accumulator.
__device__ void fused_prep(const GemmArgs& a, const int* s_sorted, const int* s_expert, int npad,
                           int epi_tid, volatile int* red) {
  const FusedPrep& P = a.prep;
  const int G = static_cast<int>(gridDim.x);
  const int cpr = P.K / 8;  // 16-byte chunks per row
  for (int p = blockIdx.x; p < npad; p += G) {
    const int sid = s_sorted[p];
    if (epi_tid == 0) P.sorted_ids[p] = sid;
    if (sid >= a.MK) {  // padding: only the sentinel exponent (uniform branch)
      if (epi_tid == 0) P.rowexp[p] = kPadRowExp;
      continue;
    }
    const uint16_t* xr = P.x + static_cast<long long>(sid / P.topk) * P.K;
    const uint4* src = reinterpret_cast<const uint4*>(xr);
    // every load of the row issued at once (rows up to kPrepChunks * 128 * 8
    // elements stay in registers; longer ones are read again below)
    constexpr int kPrepChunks = 8;
    uint4 v[kPrepChunks];
#pragma unroll
    for (int i = 0; i < kPrepChunks; ++i) {
      const int ch = epi_tid + i * kEpiThreads;
      v[i] = ch < cpr ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kPrepChunks; ++i) m = max(m, bf16x8_absmax_bits(v[i]));
    for (int ch = epi_tid + kPrepChunks * kEpiThreads; ch < cpr; ch += kEpiThreads)
      m = max(m, bf16x8_absmax_bits(src[ch]));
    m = __reduce_max_sync(0xffffffffu, m);
    if ((epi_tid & 31) == 0) red[epi_tid >> 5] = static_cast<int>(m);
    named_bar_sync(kEpiBar, kEpiThreads);
    const uint32_t mm = max(max(static_cast<uint32_t>(red[0]), static_cast<uint32_t>(red[1])),
                            max(static_cast<uint32_t>(red[2]), static_cast<uint32_t>(red[3])));
    named_bar_sync(kEpiBar, kEpiThreads);  // (red is reused by the next row)
    const int e = row_exponent(mm);
    if (epi_tid == 0) P.rowexp[p] = e;
    const float f = exp2_int(-e);
    const int32_t* pr = P.perm1 ? P.perm1 + static_cast<long long>(s_expert[p]) * P.K : nullptr;
    // chunk ch of the copy (in the packing order under act-order), as scaled fp16
    auto put = [&](int ch, uint4 x) {
      if (pr) {
        const int4 i0 = *reinterpret_cast<const int4*>(pr + 8 * ch);
        const int4 i1 = *reinterpret_cast<const int4*>(pr + 8 * ch + 4);
        x = make_uint4(bf16_pair(xr, i0.x, i0.y), bf16_pair(xr, i0.z, i0.w), bf16_pair(xr, i1.x, i1.y),
                       bf16_pair(xr, i1.z, i1.w));
      }
      const uint4 o = make_uint4(bf16x2_to_f16x2_scaled(x.x, f), bf16x2_to_f16x2_scaled(x.y, f),
                                 bf16x2_to_f16x2_scaled(x.z, f), bf16x2_to_f16x2_scaled(x.w, f));
      *reinterpret_cast<uint4*>(P.xs + b_operand_offset(ch, p, a.Gcap)) = o;
    };
#pragma unroll
    for (int i = 0; i < kPrepChunks; ++i) {
      const int ch = epi_tid + i * kEpiThreads;
      if (ch < cpr) put(ch, v[i]);
    }
    for (int ch = epi_tid + kPrepChunks * kEpiThreads; ch < cpr; ch += kEpiThreads) put(ch, src[ch]);
  }
  float4* acc4 = reinterpret_cast<float4*>(P.acc);
  for (long long i = static_cast<long long>(blockIdx.x) * kEpiThreads + epi_tid; i < P.acc_elems / 4;
       i += static_cast<long long>(G) * kEpiThreads)
    acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// kMode 1: gate/up + SwiGLU; 2: down + weighted scatter-add; 3: both in one
// launch for a small batch (phase 1 with `a`, then phase 2 with `a2`; see below).
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const GemmArgs a, const GemmArgs a2) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sStage = base + kSmStage, sRings = base + kSmRings;
  const uint32_t sBar = base + kSmBar;
  auto bar = [sBar](int i) { return sBar + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kSmMisc);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gbase + kSmMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(gbase + kSmMisc + 8);
  int* ng_max_sm = reinterpret_cast<int*>(gbase + kSmMisc + 12);
  volatile int* epi_ok = reinterpret_cast<volatile int*>(gbase + kSmMisc + 16);  // [2][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wait_ns = a.wait_kcycles;  // (the wait limit, in units of 1024 cycles)
  // Phases of this launch. The fused launch (small batches only) runs every
  // role's gate/up share and then its down share with the rings, stage counters
  // and accumulator buffers carried across: a CTA's down-projection weights
  // stream in as soon as its gate/up weights are issued, and its down
  // activations (the intermediate h) are waited for per token tile, on counters
  // the gate/up epilogues raise as they store h -- the CTAs of the grid are all
  // resident (cooperative launch), and no gate/up work ever waits on down work.
  constexpr int kPh0 = kMode == 2 ? 2 : 1, kPh1 = kMode == 1 ? 1 : 2;
  auto args = [&](int ph) -> const GemmArgs& { return (kMode == 3 && ph == 2) ? a2 : a; };
  if (threadIdx.x == 0) TRACE_POINT(13, 0);  // kernel entry
  if (threadIdx.x == 0) CTA_STAMP(0);
  // A small batch (at most 32 routed slots, small_ids set) recomputes its routing
  // tiles from the caller's topk_ids in the activation producer's warp, while
  // thread 0 initialises the barriers and warp 2 allocates tensor memory.
  const bool small = a.small_ids != nullptr;
  TokenTile* small_tiles = reinterpret_cast<TokenTile*>(gbase + kSmSmall);
  int* small_ntiles = reinterpret_cast<int*>(gbase + kSmSmall + kSmallTiles * 16);
  if (small && warp == kWarpB) {
    const SmallRoute r = small_route(a.small_ids, a.MK, a.E, kRowGroup, kBNMax, lane, a.e_begin, a.E_total);
    if (r.leader && r.tile0 < kSmallTiles) {  // one tile per expert present
      TokenTile tt;
      tt.expert = r.e;
      tt.g0 = r.seg / kRowGroup;
      tt.ngroups = r.pad / kRowGroup;
      tt.first = r.tile0;
      small_tiles[r.tile0] = tt;
    }
    const int ng = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(r.leader ? r.pad / kRowGroup : 1));
    if (lane == 0) {
      *small_ntiles = r.tot_tiles < kSmallTiles ? r.tot_tiles : kSmallTiles;
      *ng_max_sm = ng;  // the widest tile of the batch (at most 2 row groups)
    }
    if (kMode == 3) {
      // the fused launch prepares its own operand rows: the padded row list (slot
      // of every expert-sorted row, or the sentinel) and each real row's expert
      int* s_sorted = reinterpret_cast<int*>(gbase + kSmSeg);
      int* s_expert = s_sorted + kSmallPadRows;
      const int npad = r.tot_pad < kSmallPadRows ? r.tot_pad : kSmallPadRows;
      for (int p = lane; p < npad; p += 32) s_sorted[p] = a.MK;
      __syncwarp();
      if (r.e >= 0 && r.seg + r.rank < kSmallPadRows) {
        s_sorted[r.seg + r.rank] = lane;
        s_expert[r.seg + r.rank] = r.e;
      }
      if (lane == 0) {
        small_ntiles[1] = npad;
        if (r.any_bad && blockIdx.x == 0) atomicOr(a.status, kStatusBadId);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxNWS; ++i) {
      mbar_init(bar(kBarWFull + i), 1);
      mbar_init(bar(kBarWEmpty + i), 4 * kWChunk);  // 4 quadrant warps x steps
    }
    for (int i = 0; i < kNSMax; ++i) {
      mbar_init(bar(kBarFull + i), 4);
      mbar_init(bar(kBarEmpty + i), 1);
    }
    for (int i = 0; i < kMaxNB; ++i) {
      mbar_init(bar(kBarBFull + i), 1);
      mbar_init(bar(kBarBEmpty + i), 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(kBarAccFull + i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarAccEmpty + i), kEpiWarps);
      mbar_init(bar(kBarDrain + i), 1);
    }
    mbar_init(bar(kBarNever), 1);
    *abort_flag = 0;
    *last_flag = 0;
    if (!small) *ng_max_sm = 1;
    fence_mbar_init();
  }
  if (warp == kWarpMma0) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // Programmatic dependent launch. The general path waits for the preceding
  // kernel here (the routing tiles are among its outputs), then lets the next one
  // launch as this grid's CTAs retire. Starting the weight stream before that
  // wait was measured on this path: the early weight traffic slowed the
  // preceding kernel's last CTAs more than it saved.
  // A small batch (at most 32 routed slots, small_ids set) instead recomputes its
  // routing tiles here from the caller's topk_ids: one warp, one load. Only the
  // activation producer and the epilogue read the preceding kernel's outputs, so
  // only they wait; the weight stream starts right away (it has a whole decode
  // step's latency to hide and the preceding kernels are small).
  int num_tiles;
  if (small) {
    num_tiles = *small_ntiles;  // (written before the barrier above)
  } else {
    pdl_wait();
    num_tiles = a.hdr[kHdrNumTiles];
  }
  if (threadIdx.x == 0) TRACE_POINT(13, 1);
  if (threadIdx.x == 0) CTA_STAMP(1);
  int* status = a.status;
  const int G = static_cast<int>(gridDim.x);
  // Cost-weighted boundaries when the align kernel wrote them (else an even split
  // of the steps). Every CTA checks the whole table -- it starts at 0, ends at the
  // step count and never decreases -- and all of them fall back to the even split
  // (and flag the status word) if it does not: the split units' tickets rely on
  // every CTA seeing the same boundaries. (Separate launches only: a small batch
  // has no table.)
  bool weighted = kMode != 3 && a.sched != nullptr && ((a.hdr[kHdrSched] >> ((kMode & 3) - 1)) & 1) != 0;
  long long* sched_sm = reinterpret_cast<long long*>(gbase + kSmSched);
  if (weighted) {
    const long long W_total = static_cast<long long>(num_tiles) * a.R * a.KBn;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) sched_sm[i] = a.sched[i];
    __syncthreads();
    bool ok = true;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) {
      const long long v = sched_sm[i];
      ok = ok && v >= 0 && v <= W_total && (i < G ? v <= sched_sm[i + 1] : v == W_total) &&
           (i > 0 || v == 0);
    }
    weighted = __syncthreads_and(ok) != 0;
    if (!weighted && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatusBadSched);
  }
  // The split of phase ph's steps. In the fused launch the gate/up shares start
  // at multiples of 4 steps, so that every CTA's gate/up share is a whole number
  // of 2-step weight chunks (its down share starts a chunk of its own) and of
  // activation-producer rounds (each producer lane keeps its slots).
  auto phase_sched = [&](int ph) -> Sched {
    const GemmArgs& A = args(ph);
    return Sched{static_cast<long long>(num_tiles) * A.R * A.KBn, G, weighted ? sched_sm : nullptr,
                 (kMode == 3 && ph == 1) ? 4 : 1};
  };
  // this CTA's share of each phase, and where the down share starts in the CTA's
  // step sequence (every ring slot and stage follows that sequence)
  long long my_begin = 0, my_end = 0, n_first = 0;
  {
    const Sched s0 = phase_sched(kPh0);
    my_begin = s0.start(blockIdx.x);
    my_end = s0.start(blockIdx.x + 1);
    n_first = my_end - my_begin;
  }
  long long my_begin2 = 0, my_end2 = 0;
  if (kMode == 3) {
    const Sched s1 = phase_sched(2);
    my_begin2 = s1.start(blockIdx.x);
    my_end2 = s1.start(blockIdx.x + 1);
  }
  const long long n_total = n_first + (my_end2 - my_begin2);
  pdl_launch_dependents();
  if (threadIdx.x == 0) TRACE_POINT(13, 2);  // range known

  // decode this CTA's units in parallel (one round of global loads for all); the
  // widest token tile among them sizes the rings
  Unit* seg_tab = reinterpret_cast<Unit*>(gbase + kSmSeg);
  const long long u_first = my_begin / a.KBn;
  const long long n_units = my_end > my_begin ? (my_end - 1) / a.KBn - u_first + 1 : 0;
  // (a small batch needs no table: its units decode from the shared tile list)
  const int n_tab = small ? 0 : static_cast<int>(n_units < kMaxSegs ? n_units : kMaxSegs);
  if (!small) {
    if (n_units > kMaxSegs && threadIdx.x == 0) *ng_max_sm = kBNMax / kRowGroup;
    for (int i = threadIdx.x; i < n_tab; i += blockDim.x) {
      const Unit un = decode_unit(u_first + i, a.R, a.tiles, a.expert_tiles);
      seg_tab[i] = un;
      atomicMax(ng_max_sm, un.ng);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) TRACE_POINT(13, 3);  // units decoded
  // unit tables of the phases (the second only in the fused launch, always small)
  auto phase_segs = [&](int ph) -> SegTable {
    const GemmArgs& A = args(ph);
    return SegTable{seg_tab, u_first, (kMode == 3 && ph == 2) ? 0 : n_tab, A.R, A.tiles, A.expert_tiles,
                    small ? small_tiles : nullptr};
  };
  // phase ph's share [begin, end) and its first index in the CTA's step sequence
  auto phase_range = [&](int ph, long long& b, long long& e, long long& off) {
    if (kMode == 3 && ph == 2) {
      b = my_begin2;
      e = my_end2;
      off = n_first;
    } else {
      b = my_begin;
      e = my_end;
      off = 0;
    }
  };
  // (the four configurations are compile-time constants; pick one without dividing)
  const int ngm = *ng_max_sm;
  const RingCfg rc = ngm <= 1 ? ring_cfg(1) : ngm == 2 ? ring_cfg(2) : ngm == 3 ? ring_cfg(3) : ring_cfg(4);
  const int nws = rc.nws, nb = rc.nb;
  const uint32_t sW = sRings, sB = sRings + static_cast<uint32_t>(nws) * kWChunkBytes;
  // tensor memory: nst A stages, then 4 accumulators of accw columns (computed
  // in the roles that use them, from the widest tile's row groups)
#define MOE_TMEM_NST (ngm <= 2 ? static_cast<uint32_t>(kNSNarrow) : static_cast<uint32_t>(kNS))
#define MOE_TMEM_ACCW (static_cast<uint32_t>(ngm < 1 ? 1 : (ngm > 4 ? 4 : ngm)) * kRowGroup)

  if (warp == kWarpW) {
    // ------------------------------------------------ packed-weight producer
    // One lane streams the weight blocks in chunks of kWChunk consecutive steps:
    // a row tile's k-blocks are contiguous, so a chunk is one 18 KB bulk copy (one
    // per contiguous run where a chunk crosses units). Copies this large keep HBM
    // busy from a single issuing thread; 4.5 KB ones do not.
    long long c_all = 0;  // chunks issued, over the phases
    if (lane == 0) {
      // The weights are read exactly once: stream them through L2 with an
      // evict-first policy, so they do not displace the activations (re-read by
      // every row tile of their expert) or the intermediate.
      const uint64_t w_policy = l2_policy_evict_first();
      TRACE_POINT(13, 4);  // weight producer ready
      int s = 0;
      uint32_t sph = 0;  // slot of the next chunk, and the parity of its phase
      bool ok = true;
#pragma unroll
      for (int ph = kPh0; ph <= kPh1; ++ph) {
        if (!ok) break;
        const GemmArgs& A = args(ph);
        long long pb, pe, off;
        phase_range(ph, pb, pe, off);
        const long long n_it = pe - pb;
        const long long n_chunks = (n_it + kWChunk - 1) / kWChunk;
        Cursor cur(pb, pe, A.KBn, phase_segs(ph));
        for (long long c = 0; c < n_chunks; ++c) {
          if (!mbar_wait(bar(kBarWEmpty + s), sph ^ 1, abort_flag, status, kStatusTimeout, wait_ns)) {
            ok = false;
            break;
          }
          const long long it0 = c * kWChunk;
          const long long it1 = it0 + kWChunk < n_it ? it0 + kWChunk : n_it;
          TRACE_POINT(0, off + it0);
          mbar_arrive_expect_tx(bar(kBarWFull + s), static_cast<uint32_t>(it1 - it0) * kWStepBytes);
          for (long long it = it0; it < it1;) {
            int kb = 0;
            cur.seek(it, kb);
            const long long left_in_unit = cur.kb1 - kb;
            const int run = static_cast<int>(it1 - it < left_in_unit ? it1 - it : left_in_unit);
            const long long woff =
                ((static_cast<long long>(cur.un.e) * A.R + cur.un.rt) * A.KBn + kb) * kWStepBytes;
            if (MOE_CHECK(woff >= 0 && woff + static_cast<long long>(run) * kWStepBytes <= A.wpack_bytes &&
                              cur.un.e >= 0 && cur.un.e < A.E && cur.un.rt < A.R && kb + run <= A.KBn &&
                              run >= 1 && (it - it0) + run <= kWChunk,
                          A.status, A.dbg, 1, woff, run * 100 + (it - it0)))
              bulk_g2s_hint(sW + s * kWChunkBytes + static_cast<uint32_t>(it - it0) * kWStepBytes,
                            A.wpack + woff, static_cast<uint32_t>(run) * kWStepBytes,
                            bar(kBarWFull + s), w_policy);
            it += run;
          }
          ++c_all;
          if (++s == nws) {
            s = 0;
            sph ^= 1u;
          }
        }
      }
    }
    if (lane == 0) {
      // let the last chunks land before shared memory is released
      for (long long j = 0; j < nws && j < c_all; ++j) {
        const long long idx = c_all - 1 - j;
        mbar_wait_drain(bar(kBarWFull + static_cast<int>(idx % nws)),
                        static_cast<uint32_t>((idx / nws) & 1));
      }
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------ activation (B operand) producer
    // kProducerLanes lanes walk consecutive k-blocks in step and issue their
    // (2-8 KB) copies in one go: a bulk-copy issue holds its thread
    // for a while, so small copies must leave several at a time.
    // the activations are the preceding kernel's output, or, in the fused launch,
    // the rows every CTA prepares (counted on the handle's prep counter)
    bool prep_ok = true;
    if (kMode == 3) {
      if (lane < kProducerLanes)
        prep_ok = wait_counters(a.prep.fsync + kFsPrep, 1, G, abort_flag, status, wait_ns);
    } else if (small) {
      pdl_wait();
    }
    if (lane == 0) CTA_STAMP(2);
    if (lane < kProducerLanes) {
      // (indices below are in the CTA's step sequence over the phases; a down
      // share starts at a multiple of kProducerLanes, so lane l keeps the steps
      // l, l + 4, ... and its slot keeps advancing by 4 across the phases)
      long long last = -1;
      long long issued_hi = 0;  // no lane has issued a step at or beyond this index
      uint32_t mine = 0;
      int s = lane;      // slot of this lane's step, advanced by kProducerLanes (nb is a multiple)
      uint32_t sph = 0;  // parity of that slot's phase
      bool ok_all = prep_ok;
      int ready_tile = -1;  // fused down phase: the token tile whose intermediate was seen complete
#pragma unroll
      for (int ph = kPh0; ph <= kPh1; ++ph) {
        if (!ok_all) break;
        const GemmArgs& A = args(ph);
        long long pb, pe, off;
        phase_range(ph, pb, pe, off);
        const long long n_it = pe - pb;
        Cursor cur(pb, pe, A.KBn, phase_segs(ph));
        for (long long base_it = 0; base_it < n_it; base_it += kProducerLanes) {
          const long long it = base_it + lane;
          issued_hi = off + (base_it + kProducerLanes < n_it ? base_it + kProducerLanes : n_it);
          const unsigned active = __ballot_sync(0x0000000fu, it < n_it) & 0xFu;
          if (it < n_it) {
            int kb = 0;
            cur.seek(it, kb);
            if (!MOE_CHECK(cur.un.ng >= 1 && cur.un.ng <= kBNMax / 16 &&
                               static_cast<uint32_t>(cur.un.ng) * kRowGroupBytes <= rc.b_plane &&
                               cur.un.e >= 0 && cur.un.e < A.E &&
                               cur.un.g0 >= 0 && cur.un.g0 + cur.un.ng <= A.tiles_cap && kb >= 0 && kb < A.KBn,
                           A.status, A.dbg, 11, cur.un.ng * 1000 + cur.un.e, cur.un.g0 * 1000 + kb))
              cur.un.ng = 1;
            bool ok = true;
            if (kMode == 3 && ph == 2) {
              // the down GEMM's activations are the gate/up GEMM's intermediate:
              // wait (once per token tile) until every row tile of it is stored
              const int t = static_cast<int>(cur.u / A.R);
              if (t != ready_tile) {
                if (ready_tile < 0) CTA_STAMP(8);
                ok = wait_counters(a.h_ready + static_cast<long long>(t) * A.KBn, A.KBn, 2, abort_flag,
                                   status, wait_ns);
                if (ready_tile < 0) CTA_STAMP(9);
                ready_tile = t;
              }
            }
            ok = ok && mbar_wait(bar(kBarBEmpty + s), sph ^ 1, abort_flag, status, kStatusTimeout, wait_ns);
            __syncwarp(active);
            if (ok) {
              // the step's two 64-element k-blocks are two planes of the blocked layout
              const uint32_t bytes = static_cast<uint32_t>(cur.un.ng) * kRowGroupBytes;
              const long long boff =
                  (static_cast<long long>(kb) * kSub * A.Gcap + cur.un.g0) * kRowGroupBytes;
              const long long plane = static_cast<long long>(A.Gcap) * kRowGroupBytes;
              TRACE_POINT(1, off + it);
              mbar_arrive_expect_tx(bar(kBarBFull + s), kSub * bytes);
              if (MOE_CHECK(boff >= 0 && boff + bytes <= A.bsrc_bytes && bytes <= rc.b_plane && bytes > 0 &&
                                s >= 0 && s < nb,
                            A.status, A.dbg, 2, boff, bytes))
                bulk_g2s(sB + s * rc.b_stage, A.bsrc + boff, bytes, bar(kBarBFull + s));
              if (MOE_CHECK(boff + plane + bytes <= A.bsrc_bytes, A.status, A.dbg, 3, boff + plane,
                            bytes))
                bulk_g2s(sB + s * rc.b_stage + rc.b_plane, A.bsrc + boff + plane, bytes,
                         bar(kBarBFull + s));
              last = off + it;
              ++mine;
            }
            if (__any_sync(active, !ok)) {
              ok_all = false;
              break;
            }
          }
          s += kProducerLanes;
          if (s >= nb) {
            s -= nb;
            sph ^= 1u;
          }
        }
      }
      // bounded wait for this lane's last copies to land before shared memory is
      // released
      // (exactly the copies of the last nb steps issued: no later copy reused
      // their slots, so their phases cannot alias; earlier ones were consumed)
      for (long long idx = last; mine > 0 && idx >= 0 && idx + nb >= issued_hi;
           idx -= kProducerLanes) {
        mbar_wait_drain(bar(kBarBFull + static_cast<int>(idx % nb)),
                        static_cast<uint32_t>((idx / nb) & 1));
      }
    }
  } else if (warp == kWarpMma0 || warp == kWarpMma1) {
    // ------------------------------------------------ MMA issuers
    // Two warps issue alternate k-blocks of every unit into separate accumulators
    // (the epilogue adds them), so one issuer's waits and commits overlap the
    // other's MMAs. Each warp runs its loop uniformly; one elected lane issues.
    const uint32_t par = static_cast<uint32_t>(warp - kWarpMma0);
    uint32_t it_base = 0, acc_it = 0;
    bool ok = true;
    const uint64_t b_desc0 = sw128_kmajor_desc(sB);
    // B slot of this issuer's next step (its steps are 2 apart; nb is even) and
    // the parity of that slot's phase
    uint32_t sb = par, bph = 0;
    uint32_t sa = par, aph = 0;  // the same for the A stage ring (nst stages, even)
    const uint32_t nst = MOE_TMEM_NST, accw = MOE_TMEM_ACCW, acc_col0 = nst * kACols;
#pragma unroll
    for (int ph = kPh0; ph <= kPh1; ++ph) {
      if (!ok) break;
      const GemmArgs& A = args(ph);
      long long pb, pe, off;
      phase_range(ph, pb, pe, off);
      SegIter si(pb, pe, A.KBn);
      const SegTable segs = phase_segs(ph);
      long long u;
      int kb0, kb1;
      while (ok && si.next(u, kb0, kb1)) {
        const uint32_t len = static_cast<uint32_t>(kb1 - kb0);
        const uint32_t first = it_base + (((it_base & 1u) != par) ? 1u : 0u);
        const int ab = acc_it & 1;
        if (first < it_base + len) {
          Unit un = segs.get(u);
          if (!MOE_CHECK(un.ng >= 1 && un.ng <= kBNMax / 16, A.status, A.dbg, 12, un.ng, u)) un.ng = 1;
          const uint32_t idesc = idesc_f16_f32(kBM, un.ng * kRowGroup);
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarAccEmpty + ab),
                                                      ((acc_it >> 1) & 1) ^ 1, abort_flag, status,
                                                      kStatusTimeout, wait_ns));
          if (!ok) break;
          const uint32_t d_tmem = tmem + acc_col0 + (par * 2 + ab) * accw;
          uint32_t acc_flag = 0;
          for (uint32_t it = first; it < it_base + len; it += 2) {
            const uint32_t st = sa;
            if (lane == 0) TRACE_POINT(2, it);
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarBFull + sb), bph, abort_flag, status,
                                                        kStatusTimeout, wait_ns));
            if (ok)
              ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarFull + st), aph, abort_flag, status,
                                                          kStatusTimeout, wait_ns));
            if (!ok) break;
            if (lane == 0) TRACE_POINT(3, it);
            if (lane == 0 && it < 2) CTA_STAMP(4);
            if (lane == 0 && ph == 2 && kMode == 3 && it < n_first + 2) CTA_STAMP(11);
            const uint32_t a_tmem = tmem + st * kACols;
            // B stage sb is sb * b_stage bytes after stage 0, its second 64-element
            // half b_plane bytes further (16-byte units in the descriptor); +32 bytes of
            // K per MMA inside the 128-byte swizzled rows.
            const uint64_t b_desc = b_desc0 + ((sb * rc.b_stage) >> 4);
            const uint64_t b_desc1 = b_desc + (rc.b_plane >> 4);
            if (elect_one()) {
              tc_fence_after();
              tc_mma_ts(d_tmem, a_tmem, b_desc, idesc, acc_flag);
              tc_mma_ts(d_tmem, a_tmem + 8, b_desc + 2, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 16, b_desc + 4, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 24, b_desc + 6, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 32, b_desc1, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 40, b_desc1 + 2, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 48, b_desc1 + 4, idesc, 1u);
              tc_mma_ts(d_tmem, a_tmem + 56, b_desc1 + 6, idesc, 1u);
              tc_commit(bar(kBarEmpty + st));
              tc_commit(bar(kBarBEmpty + sb));
              TRACE_POINT(4, it);
              CTA_STAMP(5);
              if (ph == 1) CTA_STAMP(10);
            }
            acc_flag = 1u;
            sb += 2;
            if (sb >= static_cast<uint32_t>(nb)) {
              sb -= static_cast<uint32_t>(nb);
              bph ^= 1u;
            }
            sa += 2;
            if (sa >= nst) {
              sa -= nst;
              aph ^= 1u;
            }
          }
          if (!ok) break;
          if (elect_one()) {
            tc_commit(bar(kBarAccFull + par * 2 + ab));
            TRACE_POINT(14, 32 + acc_it * 2 + par);  // issuer done with a segment
          }
          __syncwarp();
        }
        it_base += len;
        ++acc_it;
      }
    }
    if (elect_one()) {
      tc_commit(bar(kBarDrain + par));
      mbar_wait_drain(bar(kBarDrain + par), 0);
    }
    __syncwarp();
  } else if (warp >= kWarpDeq0 && warp < kWarpEpi0) {
    // ------------------------------------------------ dequantisation into tensor memory
    // Warp (quad, phase) converts rows 32*quad .. +31 of the steps whose index in
    // this CTA's sequence is phase, phase + kDeqPhases, ... (only the index matters
    // here: it fixes the weight-ring slot and the operand stage). A step's two
    // 32-column stores are retired (wait::st + arrival) right after they are
    // issued, so the step's MMAs run while the warp converts its next step.
    const int quad = warp & 3;
    const int phase = (warp - kWarpDeq0) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t n_it = static_cast<uint32_t>(n_total);  // (the phases' steps, in sequence)
    // weight chunk of the step (2 steps per chunk): its ring slot and phase parity,
    // advanced by 2 chunks per iteration
    uint32_t ws = static_cast<uint32_t>(phase) >> 1, wpar = 0;
    // A stage of the step and the parity of that stage's use, advanced by
    // kDeqPhases steps per iteration (kDeqPhases <= nst)
    uint32_t st = static_cast<uint32_t>(phase), sph = 0;
    const uint32_t nst = MOE_TMEM_NST;
    for (uint32_t it = static_cast<uint32_t>(phase); it < n_it; it += kDeqPhases) {
      // non-blocking test of the stage-free barrier now; its latency overlaps the
      // conversion and the blocking wait below runs only if it was not ready
      const bool e_early = mbar_test_wait(bar(kBarEmpty + st), sph ^ 1);
      if (lane == 0 && quad == 0) TRACE_POINT(12, it);
      bool w_ok = mbar_wait(bar(kBarWFull + ws), wpar, abort_flag, status, kStatusTimeout, wait_ns);
      if (!__all_sync(0xffffffffu, w_ok)) break;
      if (lane == 0 && quad == 0) TRACE_POINT(5, it);
      if (lane == 0 && it == 0) CTA_STAMP(3);
      // the step's weights: slot ws, step (it & 1) of the chunk
      const uint32_t wstep = ws * kWChunk + (it & 1);
      const uint32_t wb = sW + wstep * kWStepBytes + r * 16;
      const uint32_t wsc = sW + wstep * kWStepBytes + kWCodeBytes + r * 4;
      const uint4 q0 = ld_shared_v4(wb);
      const uint4 q1 = ld_shared_v4(wb + 2048);
      const uint4 q2 = ld_shared_v4(wb + kWBlockBytes);
      const uint4 q3 = ld_shared_v4(wb + kWBlockBytes + 2048);
      const uint32_t sc0 = ld_shared_u32(wsc);  // fp16 scales of the two groups
      const uint32_t sc1 = ld_shared_u32(wsc + kWBlockBytes);
      uint32_t out[32];
      dequant_group(q0, __byte_perm(sc0, 0, 0x1010), &out[0]);
      dequant_group(q1, __byte_perm(sc0, 0, 0x3232), &out[16]);
      if (!__all_sync(0xffffffffu, e_early)) {
        w_ok = mbar_wait(bar(kBarEmpty + st), sph ^ 1, abort_flag, status, kStatusTimeout, wait_ns);
        if (!__all_sync(0xffffffffu, w_ok)) break;
      }
      if (lane == 0 && quad == 0) TRACE_POINT(7, it);
      tc_fence_after();
      __syncwarp();
      tmem_st32(a_lane + st * kACols, out);
      dequant_group(q2, __byte_perm(sc1, 0, 0x1010), &out[0]);
      dequant_group(q3, __byte_perm(sc1, 0, 0x3232), &out[16]);
      // converge before the warp-collective store; every lane has also consumed
      // its shared-memory words by now, so the slot can be released after it
      __syncwarp();
      tmem_st32(a_lane + st * kACols + 32, out);
      if (lane == 0 && quad == 0) TRACE_POINT(6, it);
      if (lane == 0) mbar_arrive(bar(kBarWEmpty + ws));
      __syncwarp();  // tcgen05.wait is warp-collective: converge after the lane-0 arrival
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) TRACE_POINT(8 + quad, it);
      if (lane == 0) mbar_arrive(bar(kBarFull + st));
      st += kDeqPhases;
      if (st >= nst) {
        st -= nst;
        sph ^= 1u;
      }
      ws += 2;
      if (ws >= static_cast<uint32_t>(nws)) {
        ws -= static_cast<uint32_t>(nws);
        wpar ^= 1u;
      }
    }
  } else if (warp >= kWarpEpi0) {
    // ------------------------------------------------ epilogue
    if (kMode == 3) {
      // prepare this CTA's rows, count it, and wait until every CTA has
      const int* s_sorted = reinterpret_cast<const int*>(gbase + kSmSeg);
      fused_prep(a, s_sorted, s_sorted + kSmallPadRows, small_ntiles[1], threadIdx.x - kWarpEpi0 * 32,
                 epi_ok + 8);
      __threadfence();
      named_bar_sync(kEpiBar, kEpiThreads);
      if (threadIdx.x == kWarpEpi0 * 32) {
        atomicAdd(a.prep.fsync + kFsPrep, 1);
        wait_counters(a.prep.fsync + kFsPrep, 1, G, abort_flag, status, wait_ns);
      }
      named_bar_sync(kEpiBar, kEpiThreads);
      __threadfence();
    } else if (small) {
      pdl_wait();  // routing rows, exponents and the zeroed accumulator / tickets
    }
    // Test hook: wait on a barrier that nothing arrives on. The wait gives up after
    // the wait limit, raises the abort flag and records the timeout; every role then
    // stops at its next wait and the teardown lets in-flight copies and MMAs land.
    if (a.test_never_wait) mbar_wait(bar(kBarNever), 0, abort_flag, a.status, kStatusTimeout, wait_ns);
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int epi_tid = threadIdx.x - kWarpEpi0 * 32;
    const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t acc_it = 0, it_base = 0, full_phase = 0;
#pragma unroll
    for (int ph = kPh0; ph <= kPh1; ++ph) {
      const GemmArgs& A = args(ph);
      const int mode = kMode == 3 ? ph : kMode;
      const Sched sc = phase_sched(ph);
      const SegTable segs = phase_segs(ph);
      long long pb, pe, off;
      phase_range(ph, pb, pe, off);
      SegIter si(pb, pe, A.KBn);
      long long u;
      int kb0, kb1;
      bool stop = false;
      while (si.next(u, kb0, kb1)) {
        Unit un = segs.get(u);
        if (!MOE_CHECK(un.ng >= 1 && un.ng <= kBNMax / 16 && un.rt >= 0 && un.rt < A.R, A.status, A.dbg,
                       13, un.ng, un.rt))
          un.ng = 1;
        const int nch = un.ng;  // 16-column chunks
        const int ab = acc_it & 1;
        const uint32_t len = static_cast<uint32_t>(kb1 - kb0);
        // which MMA issuer (even / odd k-blocks of this CTA's sequence) has a sum
        const bool has0 = len >= 2 || (it_base & 1u) == 0;
        const bool has1 = len >= 2 || (it_base & 1u) == 1;
        it_base += len;

        // routing of the tile's token rows, fetched before the wait: every row's
        // prescale exponent, and for the down GEMM its slot, token and routing
        // weight (times 2^2e, undoing the prescale of x and of h)
        int sid_r[kRowRegs], tok_r[kRowRegs], e_r[kRowRegs];
        float w_r[kRowRegs];
        {
          const int pbase = un.g0 * kRowGroup;
  #pragma unroll
          for (int j = 0; j < kRowRegs; ++j) {
            const int row = 32 * j + lane;
            const bool in_tile = row < nch * 16 &&
                                 MOE_CHECK(pbase + row < A.sorted_cap, A.status, A.dbg, 9, pbase + row, nch);
            e_r[j] = in_tile ? A.rowexp[pbase + row] : 0;  // (kPadRowExp for a padding row)
            sid_r[j] = A.MK;
            tok_r[j] = 0;
            w_r[j] = 0.f;
            if (mode == 2) {
              const int sid = in_tile ? A.sorted_ids[pbase + row] : A.MK;
              sid_r[j] = sid;
              if (sid < A.MK) {  // a real row: |e| <= kMaxRowExp
                const int e = e_r[j] < -kMaxRowExp ? -kMaxRowExp : (e_r[j] > kMaxRowExp ? kMaxRowExp : e_r[j]);
                w_r[j] = A.topk_weights[sid] * exp2_int(2 * e);
                tok_r[j] = sid / A.topk;
              }
            }
          }
        }

        bool w_ok = true;
        if (has0) {
          w_ok = mbar_wait(bar(kBarAccFull + ab), (full_phase >> ab) & 1u, abort_flag, status,
                           kStatusTimeout, wait_ns);
          full_phase ^= 1u << ab;
        }
        if (has1 && w_ok) {
          w_ok = mbar_wait(bar(kBarAccFull + 2 + ab), (full_phase >> (2 + ab)) & 1u, abort_flag,
                           status, kStatusTimeout, wait_ns);
          full_phase ^= 1u << (2 + ab);
        }
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (epi_tid == 0) TRACE_POINT(14, 512 + acc_it);  // epilogue's accumulator wait done
        if (lane == 0) epi_ok[(acc_it & 1) * 4 + quad] = w_ok ? 1 : 0;
        named_bar_sync(kEpiBar, kEpiThreads);
        const bool all_ok = epi_ok[(acc_it & 1) * 4 + 0] && epi_ok[(acc_it & 1) * 4 + 1] &&
                            epi_ok[(acc_it & 1) * 4 + 2] && epi_ok[(acc_it & 1) * 4 + 3];
        if (!all_ok) {
          stop = true;
          break;
        }
        tc_fence_after();
        const uint32_t accw = MOE_TMEM_ACCW, acc_col0 = MOE_TMEM_NST * kACols;
        const uint32_t tacc0 = tmem + t_lane + acc_col0 + ab * accw;
        const uint32_t tacc1 = tmem + t_lane + acc_col0 + (2 + ab) * accw;
        // fp32 sums of 16 token columns of this lane's row, both issuers added
        auto load_chunk = [&](int c, float (&v)[16]) {
          uint32_t rr[16];
          __syncwarp();  // tcgen05.ld is warp-collective: converge after per-lane code
  #pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
          if (has0) {
            tmem_ld16(tacc0 + c * 16, rr);
            tmem_ld_wait();
  #pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(rr[i]);
          }
          if (has1) {
            tmem_ld16(tacc1 + c * 16, rr);
            tmem_ld_wait();
  #pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += __uint_as_float(rr[i]);
          }
        };

        if (mode == 1) {
          const bool full = (kb0 == 0 && kb1 == A.KBn);
          bool write_tile = full;
          bool sat = false;
          if (full) {
            for (int c = 0; c < nch; ++c) {
              float v[16];
              load_chunk(c, v);
              if (epi_tid == 0 && c == 0) TRACE_POINT(14, 600 + acc_it * 8 + 0);  // accumulators loaded
              sat |= swiglu_chunk(v, c, quad, lane, sStage, (c >> 1) ? e_r[1] : e_r[0]);
            }
            if (epi_tid == 0) TRACE_POINT(14, 600 + acc_it * 8 + 1);  // SwiGLU staged
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarAccEmpty + ab));
          } else {
            // split unit: park this CTA's partial sums, take a ticket
            const long long ustart = u * A.KBn;
            const int part = (sc.start(blockIdx.x) < ustart) ? 1 : 0;
            float* slot = A.scratch + (static_cast<long long>(blockIdx.x) * 2 + part) * kBNMax * kBM;
            for (int c = 0; c < nch; ++c) {
              float v[16];
              load_chunk(c, v);
              const long long so = (slot - A.scratch) + (c * 16) * kBM + r;
              (void)so;  // read only by the self-checking build
              if (MOE_CHECK(so >= 0 && so + 15 * kBM < A.scratch_elems, A.status, A.dbg, 6, so, c)) {
  #pragma unroll
                for (int i = 0; i < 16; ++i) __stcg(slot + (c * 16 + i) * kBM + r, v[i]);
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarAccEmpty + ab));
            __threadfence();
            named_bar_sync(kEpiBar, kEpiThreads);
            const int c0 = sc.cta_of(ustart), c1 = sc.cta_of(ustart + A.KBn - 1);
            if (epi_tid == 0) {
              const int add = kb1 - kb0;
              const int old = atomicAdd(A.tickets + c0, add);
              *last_flag = (old + add == A.KBn) ? 1 : 0;
            }
            named_bar_sync(kEpiBar, kEpiThreads);
            if (epi_tid == 0) TRACE_POINT(14, 600 + acc_it * 8 + 5);  // ticket taken
            write_tile = *last_flag != 0;
            if (write_tile) {
              __threadfence();
              for (int c = 0; c < nch; ++c) {
                float v[16];
  #pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.f;
                for (int cc = c0; cc <= c1; ++cc) {
                  if (sc.start(cc) == sc.start(cc + 1)) continue;  // empty share: no partial
                  const int pc = (sc.start(cc) < ustart) ? 1 : 0;
                  const float* sl =
                      A.scratch + (static_cast<long long>(cc) * 2 + pc) * kBNMax * kBM;
                  const long long so = (sl - A.scratch) + (c * 16) * kBM + r;
                  (void)so;  // read only by the self-checking build
                  if (MOE_CHECK(so >= 0 && so + 15 * kBM < A.scratch_elems, A.status, A.dbg, 7, so, cc)) {
  #pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += __ldcg(sl + (c * 16 + i) * kBM + r);
                  }
                }
                sat |= swiglu_chunk(v, c, quad, lane, sStage, (c >> 1) ? e_r[1] : e_r[0]);
              }
            }
          }
          if (__any_sync(0xffffffffu, sat) && lane == 0) atomicOr(status, kStatusHSaturated);
          if (write_tile) {
            if (epi_tid == 0) TRACE_POINT(14, 600 + acc_it * 8 + 2);  // tile ready to store
            const long long hoff = (static_cast<long long>(un.rt) * A.Gcap + un.g0) * kRowGroupBytes;
            const bool hoff_ok = MOE_CHECK(hoff >= 0 && hoff + nch * kRowGroupBytes <= A.hout_bytes &&
                                               nch > 0 && nch <= kBNMax / 16,
                                           A.status, A.dbg, 5, hoff, nch);
            if (kMode == 3) {
              // The fused launch's down phase reads h from other CTAs: plain
              // stores, a fence, then the tile's counter for the k-block it
              // feeds (its two gate/up row tiles make one down k-block)
              named_bar_sync(kEpiBar, kEpiThreads);  // the staging tile is complete
              for (int i = epi_tid; i < nch * (kRowGroupBytes / 16); i += kEpiThreads)
                if (hoff_ok)
                  *reinterpret_cast<uint4*>(A.hout + hoff + i * 16) = ld_shared_v4(sStage + i * 16);
              __threadfence();
              named_bar_sync(kEpiBar, kEpiThreads);
              if (epi_tid == 0)
                atomicAdd(A.h_ready + (u / A.R) * a2.KBn + un.rt / 2, 1);
            } else {
              fence_proxy_async_smem();
              named_bar_sync(kEpiBar, kEpiThreads);
              if (epi_tid == 0) {
                if (hoff_ok) bulk_s2g(A.hout + hoff, sStage, static_cast<uint32_t>(nch) * kRowGroupBytes);
                bulk_commit();
                TRACE_POINT(14, 600 + acc_it * 8 + 3);  // bulk store issued
                bulk_wait_read_all();
                TRACE_POINT(14, 600 + acc_it * 8 + 4);  // staging tile read by the store
              }
              named_bar_sync(kEpiBar, kEpiThreads);
            }
          }
        } else {
          float* acc_col = A.acc + static_cast<long long>(un.rt) * kBM + r;
  #pragma unroll
          for (int c = 0; c < kBNMax / 16; ++c) {
            if (c < nch) {
              float v[16];
              load_chunk(c, v);
  #pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int row = c * 16 + i;
                const int sid = __shfl_sync(0xffffffffu, sid_r[row >> 5], row & 31);
                if (sid < A.MK) {
                  const int tok = __shfl_sync(0xffffffffu, tok_r[row >> 5], row & 31);
                  const float wt = __shfl_sync(0xffffffffu, w_r[row >> 5], row & 31);
                  const long long ai = (acc_col - A.acc) + static_cast<long long>(tok) * A.Kout;
                  if (MOE_CHECK(ai >= 0 && ai < A.acc_elems, A.status, A.dbg, 8, ai, sid))
                    atomicAdd(A.acc + ai, wt * v[i]);
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kBarAccEmpty + ab));
        }
        if (epi_tid == 0) TRACE_POINT(15, acc_it);  // epilogue done with a segment
        if (epi_tid == 0) CTA_STAMP(6);
        if (epi_tid == 0 && ph == 1) CTA_STAMP(12);
        ++acc_it;
      }
      if (stop) break;
    }
    if (epi_tid == 0) bulk_wait_all();
  }

  // ------------------------------------------------ teardown
  if (lane == 0) TRACE_POINT(14, warp);  // each warp reaching the teardown
  __syncwarp();  // lanes that skipped a single-lane role wait for it here
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) CTA_STAMP(7);
  if (warp == kWarpMma0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (kMode == 3) {
    // The last CTA to finish publishes the status and row counts in the workspace
    // header and clears the handle's counters for the next call.
    if (threadIdx.x == 0) {
      __threadfence();
      *last_flag = atomicAdd(a.prep.fsync + kFsExit, 1) == G - 1 ? 1 : 0;
    }
    __syncthreads();
    if (*last_flag) {
      __threadfence();
      if (threadIdx.x == 0) {
        a.prep.ws_hdr[kHdrStatus] = ld_relaxed_gpu(a.prep.fsync + kFsStatus);
        a.prep.ws_hdr[kHdrNumPadded] = small_ntiles[1];
        a.prep.ws_hdr[kHdrNumTiles] = num_tiles;
        a.prep.ws_hdr[kHdrSched] = 0;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < a.prep.fsync_words; i += blockDim.x) a.prep.fsync[i] = 0;
    }
  }
#undef MOE_TMEM_NST
#undef MOE_TMEM_ACCW
}

}  // namespace

cudaError_t gemm_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
  return e;
}

cudaError_t launch_gemm_gateup(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_k(gemm_kernel<1>, dim3(num_ctas), dim3(kThreads), kSmAlloc, stream, pdl, a, a);
}

cudaError_t launch_gemm_down(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_k(gemm_kernel<2>, dim3(num_ctas), dim3(kThreads), kSmAlloc, stream, pdl, a, a);
}

cudaError_t launch_gemm_fused(const GemmArgs& a1, const GemmArgs& a2, int num_ctas, cudaStream_t stream,
                              bool pdl) {
  return launch_k_coop(gemm_kernel<3>, dim3(num_ctas), dim3(kThreads), kSmAlloc, stream, pdl, a1, a2);
}

}  // namespace moe
