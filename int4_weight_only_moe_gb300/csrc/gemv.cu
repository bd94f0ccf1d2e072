// The two expert products of a small batch (by default at most 256 routed slots)
// on the CUDA cores: with one to four tokens per expert each product is a
// matrix-vector product, bound by the packed weight stream, so the weights are
// multiplied in registers instead of being written to tensor memory for an MMA
// whose 16-column token tile would be mostly padding.
//
//   gate/up:  [g; u] = W1[e] . x_t, epilogue h = SiLU(g) * u -> fp16 intermediate
//             (blocked layout) and h as step rows of the down product
//   down:     y = W2[e] . h_r, epilogue acc[t] += topk_weight * y (fp32 red.add)
//
// Arithmetic. The activations of every scale group of 32 reduction elements are
// 16-bit block fixed point, v = round(x * 2^e) with the group's exponent e
// chosen so that its largest |v| lies in [2^13, 2^14), written with the group's
// exact value sum V by the kernel that produces them (the routing + gather
// kernel for the hidden states, the gate/up epilogue for h). A packed word holds
// eight 4-bit codes u; a rotate and a mask turn four of them into bytes, and
// dp2a multiplies two bytes with two 16-bit values and adds, exactly, in int32.
// Per group and weight row the result is s * 2^-e * (sum u v - 8 V): the bracket
// is an exact integer below 2^23, so a group costs one fp32 rounding.
//
// Per CTA (one per SM), 24 warps, the same work on every SM sub-partition (warp
// w runs on sub-partition w % 4):
//   warps 0..15  multiply: warp (quad = w % 4, phase = w / 4) takes weight rows
//                32*quad .. +31 of the steps phase, phase + 4, ... of this CTA's
//                share, from two shared-memory rings: packed weights (10 chunks
//                of 2 steps, 18 KB bulk copies) and activation step rows with
//                their group sums (3 chunks of 8 steps, one copy per token row).
//                At the end of a unit each warp leaves its partial sums in a
//                reduction slot.
//   warps 16..19 copy producers, one per sub-partition: producer q issues the
//                activation copies of chunks q, q + 4, ... and the weight copies
//                of chunks q, q + 4, ... (the ring's first 10 weight chunks are
//                issued at the start by multiply warps 0..9, one each: they wait
//                for nothing, not even the preceding kernel), in the order of the
//                step each copy feeds. A warp that issues bulk copies slows the
//                multiply warps of its sub-partition (each copy instruction costs
//                it about 135 issue cycles, whatever its size), and the slowest
//                sub-partition sets the rings' pace: so the copies are few (a
//                chunk of 8 activation steps is one copy per row) and spread over
//                all four sub-partitions.
//   warps 20..23 epilogue: sums the 4 phases' partials in a fixed order, finishes
//                split units (gate/up: per-CTA scratch slot + ticket, summed in
//                CTA order by the last contributor), applies SiLU*up or the
//                weighted scatter-add
//
// Work split: stream-K as in the tensor-core kernel (units (tile, 128-row weight
// tile) of K/128 steps laid end to end, a contiguous share per CTA, equal in
// steps, or in cost where the tiles' row counts differ). Every wait is bounded; a wait that gives up raises the CTA's abort
// flag and records MOE_W4A16_STATUS_TIMEOUT, and every role falls through to the
// teardown, which lets the copies in flight land.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"
#include "small_route.cuh"
#include "stream_k.cuh"

namespace moe {

// Optional timeline for performance work (built with -DMOE_GEMM_TRACE): every CTA
// records global-timer stamps of a few events (latest wins), and CTA 0 per-step
// stamps of one multiply warp and of the weight producer; read back with
// moe_gemv_trace_read(). Compiled out otherwise.
#ifdef MOE_GEMM_TRACE
__device__ unsigned long long g_gv_cta[3][256][16];
__device__ unsigned long long g_gv_steps[3][8][1024];
extern "C" int moe_gemv_trace_read(unsigned long long* cta, unsigned long long* steps, int reset) {
  int e = static_cast<int>(cudaMemcpyFromSymbol(cta, g_gv_cta, sizeof(g_gv_cta)));
  if (e == 0) e = static_cast<int>(cudaMemcpyFromSymbol(steps, g_gv_steps, sizeof(g_gv_steps)));
  if (reset) {
    static unsigned long long z[3 * 8 * 1024];
    cudaMemcpyToSymbol(g_gv_cta, z, sizeof(g_gv_cta));
    cudaMemcpyToSymbol(g_gv_steps, z, sizeof(g_gv_steps));
  }
  return e;
}
__device__ __forceinline__ unsigned long long gv_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define GV_STAMP(ev) \
  do { if (blockIdx.x < 256) atomicMax(&g_gv_cta[kMode - 1][blockIdx.x][(ev)], gv_timer()); } while (0)
#define GV_POINT(slot, idx) \
  do { if (blockIdx.x == 0 && (idx) < 1024) g_gv_steps[kMode - 1][(slot)][(idx)] = gv_timer(); } while (0)
#else
#define GV_STAMP(ev) do { } while (0)
#define GV_POINT(slot, idx) do { } while (0)
#endif

namespace {

constexpr int kGvPhases = 4;                              // steps in flight (one per phase)
constexpr int kGvWarpP0 = 4 * kGvPhases;                  // 16 multiply warps, then 4 producers
constexpr int kGvWarpEpi0 = kGvWarpP0 + 4;                // then 4 epilogue warps
constexpr int kGvThreads = (kGvWarpEpi0 + 4) * 32;        // 768
constexpr int kGvEpiThreads = 128;
constexpr int kGvEpiBar = 1;                              // named barrier of the epilogue warps
constexpr int kGvRows = kGemvRows;                        // token rows of a tile
constexpr int kGvSub = 2;                                 // 64-element k-blocks per step
constexpr int kGvStepBytes = kGvSub * kWBlockBytes;       // 9 KB of packed weights
constexpr int kGvChunk = 2;                               // steps per weight copy
constexpr int kGvChunkBytes = kGvChunk * kGvStepBytes;
constexpr int kGvNWS = 10;                                // weight ring (chunks)
constexpr int kGvBSteps = 8;                              // steps per activation chunk
constexpr int kGvNB = 3;                                  // activation ring (chunks)
constexpr int kGvBRow = kGvBSteps * kXvStepBytes;         // one token row of a chunk
constexpr int kGvBStage = kGvRows * kGvBRow;              // [row][step][288 B]
// barriers
constexpr int kGbWFull = 0;                      // weight chunk landed (bulk-copy bytes)
constexpr int kGbWEmpty = kGbWFull + kGvNWS;     // weight chunk read (4 warps x 2 steps)
constexpr int kGbBFull = kGbWEmpty + kGvNWS;     // activation chunk landed
constexpr int kGbBEmpty = kGbBFull + kGvNB;      // activation chunk read (4 warps x 8 steps)
constexpr int kGbRedFull = kGbBEmpty + kGvNB;    // [2] reduction slot written (16 warps)
constexpr int kGbRedEmpty = kGbRedFull + 2;      // [2] reduction slot read (4 epilogue warps)
constexpr int kGbNever = kGbRedEmpty + 2;        // nothing arrives (the give-up test hook)
constexpr int kGvNumBars = kGbNever + 1;

using GvTile = GemvTile;  // (layout.cuh)
static_assert(sizeof(GvTile) == 32, "tile table entry size");
constexpr int kGvTileCache = kSmallTiles;  // tiles kept in shared memory (a batch's all, up to 32 slots)

// shared memory map (offsets from a 128-aligned base)
constexpr int kGsBar = 0;
constexpr int kGsMisc = kGsBar + ((kGvNumBars * 8 + 63) / 64) * 64;
// the last chunk / step copied into each ring slot (for the teardown's drain)
constexpr int kGsLast = kGsMisc + 64;  // int wlast[kGvNWS], blast[kGvNB]
// the tiles' cumulative costs, for the cost-weighted split
constexpr int kGsCum = kGsLast + (((kGvNWS + kGvNB) * 4 + 63) / 64) * 64;  // int [kGemvMaxSlots + 1]
constexpr int kGsTiles = kGsCum + (((kGemvMaxSlots + 1) * 4 + 63) / 64) * 64;
constexpr int kGsRed = kGsTiles + kSmallTiles * static_cast<int>(sizeof(GvTile));  // [2][phase][t][128] f32
constexpr int kGsBounds = kGsRed + 2 * kGvPhases * kGvRows * kBM * 4;  // int [kMaxCtas + 1]: shares
constexpr int kGsW = ((kGsBounds + (kMaxCtas + 1) * 4 + 127) / 128) * 128;
constexpr int kGsB = kGsW + kGvNWS * kGvChunkBytes;
constexpr int kGsEnd = kGsB + kGvNB * kGvBStage;
constexpr int kGsAlloc = kGsEnd + 128;  // (the base is aligned to 128 inside)
static_assert(kGsAlloc <= 227 * 1024, "shared memory budget");
static_assert(kGvStepBytes % 16 == 0 && kGvBStage % 16 == 0 && kGsB % 16 == 0, "16-byte alignment");
// Parity safety: a multiply warp sees every second weight chunk (its steps are 4
// apart, 2 steps a chunk) and, with an even ring, only slots it has itself waited
// on in their previous phase. An activation chunk is read by every multiply warp
// (each phase has 2 of its 8 steps), so none can be refilled while a warp still
// waits for it. The activation ring covers the weight ring's steps.
static_assert(kGvNWS % 2 == 0 && kGvPhases == 2 * kGvChunk && kGvPhases == 4 && kGvBSteps % kGvPhases == 0 &&
                  kGvNB * kGvBSteps >= kGvNWS * kGvChunk,
              "ring depths");

// acc + x.lo * code byte 2h + x.hi * code byte 2h + 1 (h = 0: .lo, 1: .hi): two
// exact integer products of a 16-bit activation and an unsigned 4-bit code.
__device__ __forceinline__ int dp2a_lo(uint32_t x, uint32_t codes, int acc) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(codes), "r"(acc));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t x, uint32_t codes, int acc) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(codes), "r"(acc));
  return d;
}

// One step (128 reduction elements) of weight row r for token rows T0 .. T0+T-1
// of the tile: per scale group, the exact integer sum of code x value over its 32
// elements (dp2a), minus 8 times the group's value sum, times the weight scale
// and the group's 2^-e. w: the step's packed weights; x: the step's row 0 in the
// activation stage (row t at + t * kGvBRow). A group's codes are unpacked once
// for all the tile's rows; the groups are unrolled for a single row only (more
// would not fit the 80 registers a thread of this CTA has).
template <int T, int T0>
__device__ __forceinline__ void gv_step(const uint8_t* w, const uint8_t* x, int r, float (&acc)[kGvRows]) {
  static_assert(T >= 1 && T <= 4 && T0 + T <= kGvRows, "rows per call");
#pragma unroll(T == 1 ? 4 : 1)
  for (int gi = 0; gi < 4; ++gi) {
    // group gi: half gi % 2 of the step's k-block gi / 2
    const uint8_t* blk = w + (gi >> 1) * kWBlockBytes;
    const uint4 qv = *reinterpret_cast<const uint4*>(blk + (gi & 1) * 2048 + r * 16);
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(blk + kWCodeBytes + r * 4);
    const float s = __half2float(__ushort_as_half(static_cast<uint16_t>((gi & 1) ? (sw >> 16) : (sw & 0xFFFFu))));
    const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
    int part[T];
#pragma unroll
    for (int t = 0; t < T; ++t) part[t] = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // codes of elements 2, 4, 3, 5 and 0, 7, 1, 6 as bytes (layout.cuh), each
      // times 4: the codes sit at bits 2..5 of every byte, directly or after a
      // rotation by 4, so one mask takes them (the factor 4 goes into the scale)
      const uint32_t c0 = w4[j] & 0x3C3C3C3Cu;
      const uint32_t c1 = __funnelshift_r(w4[j], w4[j], 4) & 0x3C3C3C3Cu;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + (T0 + t) * kGvBRow + gi * 64 + j * 16);
        part[t] = dp2a_lo(xv.x, c0, part[t]);
        part[t] = dp2a_hi(xv.y, c0, part[t]);
        part[t] = dp2a_lo(xv.z, c1, part[t]);
        part[t] = dp2a_hi(xv.w, c1, part[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
      // the group's header: 2^-(e+2) and 32 times its value sum V
      const int2 hdr = *reinterpret_cast<const int2*>(x + (T0 + t) * kGvBRow + 256 + gi * 8);
      // 4 sum (u - 8) v: exact in int32, and in fp32 (a multiple of 4 below 2^25);
      // times s 2^(-e-2), an exact power-of-two scaling of s, so the product is
      // s 2^-e sum (u - 8) v and the fma rounds once
      const float dot = static_cast<float>(part[t] - hdr.y);
      acc[T0 + t] = fmaf(s * __int_as_float(hdr.x), dot, acc[T0 + t]);
    }
  }
}

// The CTA's step sequence in closed form: sequence index `it` -> (unit, step of
// the unit), in SegIter's order (the unit the share starts inside, the unit it
// ends inside, then the whole units), plus the end of that unit's steps within
// the share. Any thread can map any step without walking the sequence.
struct GvSeq {
  long long u0, u1, uw, len0, len1;
  int KBn, kb00;
  __device__ GvSeq(long long begin, long long end, int kbn) : KBn(kbn) {
    u0 = begin / KBn;
    u1 = end > begin ? (end - 1) / KBn : u0;
    const bool p0 = end > begin && (begin > u0 * KBn || end < (u0 + 1) * KBn);
    const bool p1 = end > begin && u1 != u0 && end < (u1 + 1) * KBn;
    kb00 = static_cast<int>(begin - u0 * KBn);
    len0 = p0 ? ((end < (u0 + 1) * KBn ? end : (u0 + 1) * KBn) - begin) : 0;
    len1 = p1 ? end - u1 * KBn : 0;
    uw = p0 ? u0 + 1 : u0;
  }
  __device__ __forceinline__ void at(long long it, long long& u, int& kb, int& kb_end) const {
    if (it < len0) {
      u = u0;
      kb = kb00 + static_cast<int>(it);
      kb_end = kb00 + static_cast<int>(len0);
    } else if (it < len0 + len1) {
      u = u1;
      kb = static_cast<int>(it - len0);
      kb_end = static_cast<int>(len1);
    } else {
      const long long j = it - len0 - len1;
      u = uw + j / KBn;
      kb = static_cast<int>(j % KBn);
      kb_end = KBn;
    }
  }
};

// Relative cost of one step of a tile with T token rows (T = 1..4). One row is
// bound by the weight stream, more by the arithmetic. Measured at full size on 64
// experts with T rows each, a step costs 1.31, 1.66, 2.04 times the one-row step
// for T = 2, 3, 4. In a batch that mixes them the one-row shares stream faster
// than when all shares are one-row, and the best split (measured at M = 6 to 32)
// charges 1.38, 1.75, 2.19.
__host__ __device__ constexpr int gv_step_cost(int T) { return T <= 1 ? 16 : T == 2 ? 22 : T == 3 ? 28 : 35; }

// The stream-K split weighted by tile cost: every unit of tile i costs
// gv_step_cost(rows of tile i) per step, and CTA c starts at the first step at or
// after which c / G of the total cost has gone before (so shares start anywhere,
// like the even split's). cum[i] = cost of tiles 0 .. i-1 (cum[0] = 0), per step
// of a unit; a tile has unit_steps = R * KBn steps.
struct GvSched {
  const int* cum;  // [ntiles + 1], shared memory
  int ntiles, G;
  long long unit_steps;
  __device__ __forceinline__ long long total_steps() const { return ntiles * unit_steps; }
  __device__ long long start(int c) const {
    if (c <= 0) return 0;
    if (c >= G) return total_steps();
    const long long total = cum[ntiles] * unit_steps;
    const long long target = (static_cast<long long>(c) * total + G - 1) / G;  // ceil(c * total / G)
    // the tile in which the cumulative cost reaches target
    int lo = 0, hi = ntiles - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] * unit_steps <= target) lo = mid; else hi = mid - 1;
    }
    const long long base = cum[lo] * unit_steps;
    const long long per = cum[lo + 1] - cum[lo];  // this tile's cost per step
    const long long k = per > 0 ? (target - base + per - 1) / per : 0;
    const long long s = lo * unit_steps + (k < unit_steps ? k : unit_steps);
    return s < total_steps() ? s : total_steps();
  }
};

// kMode 1: gate/up + SwiGLU; 2: down + weighted scatter-add (b unused: = a);
// 3: both products of a batch of at most 32 routed slots in one launch, a = the
// gate/up product's arguments, b = the down product's. In one launch every role
// runs the gate/up share and then the down share of its CTA as one sequence of
// steps (the rings run on across the boundary), so the down product's weight
// stream follows the gate/up one without a gap; the down product's activation
// rows are the intermediate that the gate/up epilogues of the whole grid write,
// so the fourth copy producer takes them (and leaves the weight copies to the
// other three): it waits per (tile, step) for the two gate/up epilogues that
// write each step row (counters raised with a fence and an atomic add). All CTAs
// are resident together (cooperative launch).
template <int kMode>
__global__ void __launch_bounds__(kGvThreads, 1) gemv_kernel(const GemmArgs a, const GemmArgs b) {
  constexpr int kNph = kMode == 3 ? 2 : 1;  // products in this launch
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;  // (bulk copies need 16-byte alignment)
  uint8_t* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) -> uint32_t { return base + kGsBar + static_cast<uint32_t>(i) * 8u; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kGsMisc);
  volatile int* last_flag = reinterpret_cast<volatile int*>(gbase + kGsMisc + 4);
  int* ntiles_sm = reinterpret_cast<int*>(gbase + kGsMisc + 8);
  volatile int* epi_ok = reinterpret_cast<volatile int*>(gbase + kGsMisc + 16);  // [2][4]
  // (one launch) multiply warps through the gate/up steps
  volatile int* phase_a_done = reinterpret_cast<volatile int*>(gbase + kGsMisc + 56);
  GvTile* tiles = reinterpret_cast<GvTile*>(gbase + kGsTiles);
  float* red = reinterpret_cast<float*>(gbase + kGsRed);
  int* bounds = reinterpret_cast<int*>(gbase + kGsBounds);
  const uint32_t sW = base + kGsW, sB = base + kGsB;
  int* wlast = reinterpret_cast<int*>(gbase + kGsLast);
  int* blast = wlast + kGvNWS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t wait_ns = a.wait_kcycles;
  int* status = a.status;
  if (threadIdx.x == 0) GV_STAMP(0);

  // Tiles of the batch from the caller's topk_ids (warp 0): every expert's slots,
  // in the padded rows the routing + gather kernel placed them in (16 per expert
  // and row group), cut into tiles of at most 4 rows, experts in id order. A
  // larger batch reads the align kernel's tile list instead (its count now; the
  // tiles below, once the share is known): the whole kernel then waits for the
  // preceding kernels.
  const bool small = a.small_ids != nullptr;
  if (warp == 0 && !small) {
    pdl_wait();
    if (lane == 0) *ntiles_sm = a.hdr[kHdrNumGemvTiles];
  }
  if (warp == 0 && small) {
    if (a.ids_after_pdl) pdl_wait();  // the ids are the preceding kernel's output
    const int v = lane < a.MK ? a.small_ids[lane] : -1;
    const SmallRoute r = small_route_ids(v, a.MK, a.E, kRowGroup, kBNMax, lane, a.e_begin, a.E_total);
    const int nt = r.leader ? (r.cnt + kGvRows - 1) / kGvRows : 0;
    const int lead_e = r.leader ? r.e : -1;
    int t0 = 0, tot = 0;
    for (int j = 0; j < 32; ++j) {
      const int ej = __shfl_sync(0xffffffffu, lead_e, j);
      const int nj = __shfl_sync(0xffffffffu, nt, j);
      if (ej >= 0) {
        tot += nj;
        if (ej < r.e) t0 += nj;
      }
    }
    if (r.e >= 0 && r.seg + r.rank < kSmallPadRows) {
      const int ti = t0 + r.rank / kGvRows;
      if (ti < kSmallTiles) {
        GvTile& tl = tiles[ti];
        if (r.rank % kGvRows == 0) {
          tl.e = r.e;
          tl.p0 = r.seg + r.rank;
          tl.n = r.cnt - r.rank < kGvRows ? r.cnt - r.rank : kGvRows;
        }
        tl.slot[r.rank % kGvRows] = lane;
      }
    }
    if (lane == 0) *ntiles_sm = tot < kSmallTiles ? tot : kSmallTiles;
    if (lane == 0) GV_STAMP(9);
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kGvNWS; ++i) {
      mbar_init(bar(kGbWFull + i), 1);
      mbar_init(bar(kGbWEmpty + i), 4 * kGvChunk);
      wlast[i] = -1;
    }
    for (int i = 0; i < kGvNB; ++i) {
      mbar_init(bar(kGbBFull + i), 1);
      mbar_init(bar(kGbBEmpty + i), 4 * kGvBSteps);
      blast[i] = -1;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kGbRedFull + i), 4 * kGvPhases);
      mbar_init(bar(kGbRedEmpty + i), 4);
    }
    mbar_init(bar(kGbNever), 1);
    *abort_flag = 0;
    *last_flag = 0;
    *phase_a_done = 0;
    fence_mbar_init();
    GV_STAMP(10);
  }
  if (threadIdx.x == 64) GV_STAMP(11);
  __syncthreads();

  const int ntiles = *ntiles_sm;
  const int G = static_cast<int>(gridDim.x);
  // Shares: a small batch's weighted by the tiles' costs (its tiles are all in
  // shared memory); the align kernel's list split evenly.
  // (tiles of one cost, as at decode, take the even split's simpler arithmetic).
  // Costs per tile into cum[1..], then a prefix sum by warp 0.
  int* cum = reinterpret_cast<int*>(gbase + kGsCum);
  int* weighted_sm = reinterpret_cast<int*>(gbase + kGsMisc + 12);
  for (int i = threadIdx.x; i < ntiles; i += blockDim.x)
    cum[i + 1] = gv_step_cost(small ? tiles[i].n : a.gv_tiles[i].n);
  __syncthreads();
  if (warp == 0) {
    // lane l sums tiles 8l .. 8l + 7 (ntiles <= 256), then a warp scan of the lane sums
    constexpr int kPer = (kGemvMaxSlots + 31) / 32;
    int v[kPer];
    int lane_sum = 0;
    bool uneven = false;
    const int c0 = ntiles > 0 ? cum[1] : 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = lane * kPer + j;
      v[j] = i < ntiles ? cum[i + 1] : 0;
      lane_sum += v[j];
      uneven = uneven || (i < ntiles && v[j] != c0);
    }
    int incl = lane_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uneven = __any_sync(0xffffffffu, uneven);
    __syncwarp();  // (every lane has read its costs before any lane overwrites)
    if (uneven) {
      int run = incl - lane_sum;  // cost of the tiles before this lane's
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = lane * kPer + j;
        if (i < ntiles) cum[i] = run;
        run += v[j];
      }
      if (lane == 31) cum[ntiles] = incl;
    } else if (lane == 0) {
      cum[0] = 0;  // an even split: one cost unit per step of one tile spanning all
      cum[1] = 1;
    }
    if (lane == 0) *weighted_sm = uneven ? 1 : 0;
  }
  __syncthreads();
  const bool weighted = *weighted_sm != 0;
  // every CTA's first step (the host keeps the step count below 2^31), computed
  // in parallel into shared memory: the shares, and the epilogue's lookups of the
  // CTAs that share a unit, then cost nothing
  const int sc_tiles = weighted ? ntiles : 1;
  const long long sc_unit = weighted ? static_cast<long long>(a.R) * a.KBn : static_cast<long long>(ntiles) * a.R * a.KBn;
  int* shares_b = reinterpret_cast<int*>(gbase + kGsMisc + 48);  // [2] the down share (one launch)
  {
    const GvSched s0{cum, sc_tiles, G, sc_unit};
    for (int c = threadIdx.x; c <= G; c += blockDim.x) bounds[c] = static_cast<int>(s0.start(c));
    if (kMode == 3 && warp == kGvWarpEpi0) {
      // (an epilogue warp, idle here: this CTA's share of the down product)
      const GvSched s1{cum, sc_tiles, G,
                       weighted ? static_cast<long long>(b.R) * b.KBn : static_cast<long long>(ntiles) * b.R * b.KBn};
      if (lane < 2) shares_b[lane] = static_cast<int>(s1.start(static_cast<int>(blockIdx.x) + lane));
    }
  }
  __syncthreads();
  const long long my_begin = bounds[blockIdx.x], my_end = bounds[blockIdx.x + 1];
  // the CTA whose share contains step g
  auto cta_of = [&](long long g) -> int {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bounds[mid] <= g) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // this CTA's sequence: the gate/up (or the one) product's n1 steps, then in one
  // launch the down product's n_it - n1
  const long long n1 = my_end - my_begin;
  const long long b2 = kMode == 3 ? shares_b[0] : 0, e2 = kMode == 3 ? shares_b[1] : 0;
  const long long n_it = n1 + (e2 - b2);
  const GvSeq seq(my_begin, my_end, a.KBn);
  const GvSeq seq2(b2, e2, kMode == 3 ? b.KBn : a.KBn);
  // step `it` of the sequence -> product ph, unit, k-block, end of its run in the unit
  // (a run never crosses from one product to the other)
  auto step_at = [&](long long it, int& ph, long long& u, int& kb, int& kbe) {
    ph = (kMode == 3 && it >= n1) ? 1 : 0;
    if (ph)
      seq2.at(it - n1, u, kb, kbe);
    else
      seq.at(it, u, kb, kbe);
  };
  // Tiles in shared memory: all of a small batch's; for the align kernel's list
  // the window of this CTA's share (tiles beyond it, only when a CTA spans more
  // than kGvTileCache tiles, are read from global memory).
  const int t_lo = small ? 0 : static_cast<int>(my_begin / (static_cast<long long>(a.R) * a.KBn));
  if (!small) {
    for (int i = threadIdx.x; i < kGvTileCache && t_lo + i < ntiles; i += blockDim.x) tiles[i] = a.gv_tiles[t_lo + i];
    __syncthreads();
  }
  auto tile_at = [&](long long ti) -> const GvTile* {
    const long long k = ti - t_lo;
    return (k >= 0 && k < kGvTileCache) ? tiles + k : a.gv_tiles + ti;
  };
  pdl_launch_dependents();
  if (threadIdx.x == 0) GV_STAMP(1);

  const long long n_chunks = (n_it + kGvChunk - 1) / kGvChunk;
  // Copy weight chunk c (steps 2c, 2c + 1 of the sequence) into its ring slot.
  auto issue_w = [&](long long c) {
    const int s = static_cast<int>(c % kGvNWS);
    const long long it0 = c * kGvChunk;
    const long long it1 = it0 + kGvChunk < n_it ? it0 + kGvChunk : n_it;
    wlast[s] = static_cast<int>(c);
    mbar_arrive_expect_tx(bar(kGbWFull + s), static_cast<uint32_t>(it1 - it0) * kGvStepBytes);
    GV_POINT(0, c);
    if (c == 0) GV_STAMP(8);
    const uint64_t w_policy = l2_policy_evict_first();  // read once: keep L2 for the operands
    for (long long it = it0; it < it1;) {
      long long u;
      int ph, kb, kbe;
      step_at(it, ph, u, kb, kbe);
      const int run = static_cast<int>(it1 - it < kbe - kb ? it1 - it : kbe - kb);
      const int R = ph ? b.R : a.R, KBn = ph ? b.KBn : a.KBn;
      const int e = tile_at(u / R)->e;
      const int rt = static_cast<int>(u % R);
      const long long woff = ((static_cast<long long>(e) * R + rt) * KBn + kb) * kGvStepBytes;
      if (MOE_CHECK(woff >= 0 && woff + static_cast<long long>(run) * kGvStepBytes <= (ph ? b.wpack_bytes : a.wpack_bytes) &&
                        e >= 0 && e < a.E && run >= 1,
                    a.status, a.dbg, 41, woff, run))
        bulk_g2s_hint(sW + s * kGvChunkBytes + static_cast<uint32_t>(it - it0) * kGvStepBytes,
                      (ph ? b.wpack : a.wpack) + woff, static_cast<uint32_t>(run) * kGvStepBytes, bar(kGbWFull + s),
                      w_policy);
      it += run;
    }
  };

  // Activation chunks: 8 steps each, every token row of their tiles. In one
  // launch the down product's steps start a fresh chunk (pad skipped positions):
  // a chunk holding both products' steps would make the last gate/up steps of
  // the CTA wait for intermediate rows that they themselves help to finish.
  const long long nbA = (n1 + kGvBSteps - 1) / kGvBSteps;  // chunks of the first product's steps
  const long long pad = (kMode == 3 && n_it > n1) ? nbA * kGvBSteps - n1 : 0;
  auto b_chunk = [&](long long nb, long long& it0, long long& it1) {
    it0 = nb < nbA ? nb * kGvBSteps : nb * kGvBSteps - pad;
    const long long lim = nb < nbA ? n1 : n_it;
    it1 = it0 + kGvBSteps < lim ? it0 + kGvBSteps : lim;
  };
  // Copy activation chunk nb into its ring slot, once the slot is free.
  auto issue_b = [&](long long nb) {
    const int s = static_cast<int>(nb % kGvNB);
    long long it0, it1;
    b_chunk(nb, it0, it1);
    // the chunk's pieces (one per unit it touches): their bytes, then the copies
    uint32_t bytes = 0;
    for (long long it = it0; it < it1;) {
      long long u;
      int ph, kb, kbe;
      step_at(it, ph, u, kb, kbe);
      const int run = static_cast<int>(it1 - it < kbe - kb ? it1 - it : kbe - kb);
      bytes += static_cast<uint32_t>(tile_at(u / (ph ? b.R : a.R))->n * run * kXvStepBytes);
      it += run;
    }
    blast[s] = static_cast<int>(nb);
    mbar_arrive_expect_tx(bar(kGbBFull + s), bytes);
    for (long long it = it0; it < it1;) {
      long long u;
      int ph, kb, kbe;
      step_at(it, ph, u, kb, kbe);
      const int run = static_cast<int>(it1 - it < kbe - kb ? it1 - it : kbe - kb);
      const GvTile& tl = *tile_at(u / (ph ? b.R : a.R));
      const int KBn = ph ? b.KBn : a.KBn;
      for (int t = 0; t < tl.n; ++t) {
        // (step rows are indexed by the routed slot)
        const long long xoff = (static_cast<long long>(tl.slot[t]) * KBn + kb) * kXvStepBytes;
        if (MOE_CHECK(xoff >= 0 && xoff + static_cast<long long>(run) * kXvStepBytes <= (ph ? b.xv_bytes : a.xv_bytes) &&
                          tl.n <= kGvRows,
                      a.status, a.dbg, 42, xoff, run))
          bulk_g2s(sB + static_cast<uint32_t>(s) * kGvBStage + t * kGvBRow + static_cast<uint32_t>(it - it0) * kXvStepBytes,
                   (ph ? b.xv_in : a.xv_in) + xoff, static_cast<uint32_t>(run) * kXvStepBytes, bar(kGbBFull + s));
      }
      it += run;
    }
    // a gate/up chunk cut short by the padding: its missing steps' reader
    // arrivals (4 a step), so that the slot's next use finds it released
    if (kMode == 3 && pad > 0 && nb == nbA - 1)
      mbar_arrive_cnt(bar(kGbBEmpty + s), static_cast<uint32_t>(4 * (kGvBSteps - (it1 - it0))));
  };
  const long long n_bchunks = (n_it + pad + kGvBSteps - 1) / kGvBSteps;
  // (in one launch the down product's chunks are the fourth producer's)
  const long long nb_copier = kMode == 3 ? nbA : n_bchunks;

  if (warp >= kGvWarpP0 && warp < kGvWarpEpi0) {
    // ------------------------------------------------ copy producers
    if (lane == 0) {
      const int q = warp - kGvWarpP0;  // (= this warp's sub-partition)
      // Chunks go round kP producers. A producer issues an activation chunk only
      // once its weight copies have reached the chunk's steps, and a weight copy
      // waits for its slot's reader 10 chunks back: so it is never two uses of a
      // slot ahead of the readers, and a parity wait on the slot's release means
      // the latest use. In one launch the fourth producer issues no weight copies
      // and takes the down product's activation chunks, which wait for other
      // CTAs: it starts only once every multiply warp is through the gate/up
      // steps (then each slot's barrier is at a known phase, and from there on
      // only this producer refills the slots).
      constexpr int kP = kMode == 3 ? 3 : 4;
      const bool copier = kMode == 3 && q == 3;
      // activation rows: the preceding kernel's output
      bool b_ready = false;
      long long nb = copier ? n_bchunks : q, nw = copier ? n_chunks : q;  // next activation / weight chunk
      while (nw < kGvNWS) nw += kP;  // (the multiply warps copy the ring's first chunks)
      while (nb < nb_copier || nw < n_chunks) {
        // the copy feeding the earlier step first: a wait then only depends on
        // steps whose copies were issued before it
        if (nb < nb_copier && (nw >= n_chunks || nb * kGvBSteps <= nw * kGvChunk)) {
          if (!b_ready) {
            if (!a.ids_after_pdl) pdl_wait();
            if (q == 0) GV_STAMP(2);
            b_ready = true;
          }
          const int s = static_cast<int>(nb % kGvNB);
          if (!mbar_wait(bar(kGbBEmpty + s), static_cast<uint32_t>((nb / kGvNB) & 1) ^ 1u, abort_flag, status,
                         kStatusTimeout, wait_ns))
            break;
          issue_b(nb);
          nb += kP;
        } else {
          const int s = static_cast<int>(nw % kGvNWS);
          if (!mbar_wait(bar(kGbWEmpty + s), static_cast<uint32_t>((nw / kGvNWS) & 1) ^ 1u, abort_flag, status,
                         kStatusTimeout, wait_ns))
            break;
          issue_w(nw);
          nw += kP;
        }
      }
      if (copier && *abort_flag == 0 && nb_copier < n_bchunks) {
        pdl_wait();  // (the zeroed counters)
        // every multiply warp through the gate/up steps (bounded like every wait)
        const long long t0 = clock64();
        while (*phase_a_done < kGvWarpP0 && *abort_flag == 0) {
          if (((clock64() - t0) >> 10) > static_cast<long long>(wait_ns)) {
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
          }
          __nanosleep(128);
        }
        for (long long nc = nb_copier; nc < n_bchunks && *abort_flag == 0; ++nc) {
          // the chunk's down steps: wait until both gate/up epilogues of every one
          // of their step rows have stored it (per tile and step: a counter)
          bool ok = true;
          long long it0c, it1;
          b_chunk(nc, it0c, it1);
          for (long long it = it0c; ok && it < it1;) {
            long long u;
            int ph, kb, kbe;
            step_at(it, ph, u, kb, kbe);
            const int run = static_cast<int>(it1 - it < kbe - kb ? it1 - it : kbe - kb);
            const long long ti = u / b.R;
            if (ph == 1 &&
                MOE_CHECK(ti >= 0 && ti < kSmallTiles && kb + run <= b.KBn, a.status, a.dbg, 47, ti, kb))
              ok = wait_counters(b.h_ready + ti * b.KBn + kb, run, 2, abort_flag, status, wait_ns);
            it += run;
          }
          if (nc == nb_copier) GV_STAMP(12);
          const int s = static_cast<int>(nc % kGvNB);
          if (!ok || (nc >= kGvNB && !mbar_wait(bar(kGbBEmpty + s), static_cast<uint32_t>((nc / kGvNB) & 1) ^ 1u,
                                                 abort_flag, status, kStatusTimeout, wait_ns)))
            break;
          issue_b(nc);
        }
      }
    }
  } else if (warp < kGvWarpP0) {
    // ------------------------------------------------ multiply
    // the weight ring's first chunks: one copy per warp, nothing to wait for
    if (lane == 0 && warp < kGvNWS && warp < n_chunks) issue_w(warp);
    __syncwarp();
    const int quad = warp & 3;
    const int phase = warp >> 2;
    const int r = quad * 32 + lane;
    long long u;
    int kb0, kb1;
    uint32_t it_base = 0, ru = 0;
    bool ok = true;
#pragma unroll 1
    for (int ph = 0; ph < kNph; ++ph) {
    const int R = ph ? b.R : a.R;
    SegIter si(ph ? b2 : my_begin, ph ? e2 : my_end, ph ? b.KBn : a.KBn);
    while (ok && si.next(u, kb0, kb1)) {
      const uint32_t len = static_cast<uint32_t>(kb1 - kb0);
      const int T = tile_at(u / R)->n;
      float acc[kGvRows] = {0.f, 0.f, 0.f, 0.f};
      for (uint32_t it = it_base + ((static_cast<uint32_t>(phase) - it_base) & 3u); it < it_base + len;
           it += kGvPhases) {
        const uint32_t c = it >> 1;
        const uint32_t ws = c % kGvNWS, wpar = (c / kGvNWS) & 1u;
        const uint32_t vb = it + ((kMode == 3 && it >= n1) ? static_cast<uint32_t>(pad) : 0u);  // (padded)
        const uint32_t cb = vb / kGvBSteps;
        const uint32_t sb = cb % kGvNB, bpar = (cb / kGvNB) & 1u;
        bool w_ok = mbar_wait(bar(kGbWFull + ws), wpar, abort_flag, status, kStatusTimeout, wait_ns);
        if (warp == 0 && lane == 0) {
          GV_POINT(1, it >> 2);
          if (it < 4) GV_STAMP(3);
        }
        w_ok = w_ok && mbar_wait(bar(kGbBFull + sb), bpar, abort_flag, status, kStatusTimeout, wait_ns);
        if (warp == 0 && lane == 0) {
          GV_POINT(2, it >> 2);
          if (it < 4) GV_STAMP(4);
        }
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        const uint8_t* wstep = gbase + kGsW + ws * kGvChunkBytes + (it & 1u) * kGvStepBytes;
        const uint8_t* xst = gbase + kGsB + sb * kGvBStage + (vb % kGvBSteps) * kXvStepBytes;
        if (T == 1) {
          gv_step<1, 0>(wstep, xst, r, acc);
        } else {
          if (T == 2) gv_step<2, 0>(wstep, xst, r, acc);
          else if (T == 3) gv_step<3, 0>(wstep, xst, r, acc);
          else gv_step<4, 0>(wstep, xst, r, acc);
        }
        __syncwarp();  // every lane has read the step's shared memory
        if (lane == 0) {
          mbar_arrive(bar(kGbWEmpty + ws));
          mbar_arrive(bar(kGbBEmpty + sb));
        }
        if (warp == 0 && lane == 0) {
          GV_POINT(3, it >> 2);
          GV_STAMP(5);
        }
        if (warp > 0 && warp < 4 && lane == 0) GV_POINT(3 + warp, it >> 2);
      }
      if (!ok) break;
      it_base += len;
      // this warp's share of the unit's sums (zero where it had no step)
      const uint32_t rs = ru & 1u, rpar = (ru >> 1) & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kGbRedEmpty + rs), rpar ^ 1, abort_flag, status,
                                               kStatusTimeout, wait_ns)))
        break;
      float* dst = red + ((rs * kGvPhases + phase) * kGvRows) * kBM + r;
#pragma unroll
      for (int t = 0; t < kGvRows; ++t) dst[t * kBM] = acc[t];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kGbRedFull + rs));
      ++ru;
    }
    // (one launch: this warp has released every gate/up activation chunk)
    if (kMode == 3 && ph == 0 && ok && lane == 0) atomicAdd(const_cast<int*>(phase_a_done), 1);
    }
  } else {
    // ------------------------------------------------ epilogue
    pdl_wait();  // exponents, zeroed accumulator and tickets, routing weights
    // Test hook: wait on a barrier that nothing arrives on (gives up, raises the
    // abort flag and records the timeout).
    if (a.test_never_wait) mbar_wait(bar(kGbNever), 0, abort_flag, a.status, kStatusTimeout, wait_ns);
    const int tid = threadIdx.x - kGvWarpEpi0 * 32;  // = the weight row this thread sums
    const int ew = tid >> 5;
    const GemmArgs& D = kMode == 3 ? b : a;  // the down product's arguments
    long long u;
    int kb0, kb1;
    uint32_t ru = 0;
    bool sat = false, ok = true;
#pragma unroll 1
    for (int ph = 0; ph < kNph && ok; ++ph) {
    const bool down = kMode == 2 || ph == 1;
    const int R = ph ? b.R : a.R;
    SegIter si(ph ? b2 : my_begin, ph ? e2 : my_end, ph ? b.KBn : a.KBn);
    while (si.next(u, kb0, kb1)) {
      const GvTile& tl = *tile_at(u / R);
      const int T = tl.n;
      const int rt = static_cast<int>(u % R);
      const uint32_t rs = ru & 1u, rpar = (ru >> 1) & 1u;
      const bool w_ok = __all_sync(0xffffffffu, mbar_wait(bar(kGbRedFull + rs), rpar, abort_flag, status,
                                                          kStatusTimeout, wait_ns));
      if (lane == 0) epi_ok[(ru & 1u) * 4 + ew] = w_ok ? 1 : 0;
      named_bar_sync(kGvEpiBar, kGvEpiThreads);
      const bool all_ok = epi_ok[(ru & 1u) * 4 + 0] && epi_ok[(ru & 1u) * 4 + 1] &&
                          epi_ok[(ru & 1u) * 4 + 2] && epi_ok[(ru & 1u) * 4 + 3];
      if (!all_ok) {
        ok = false;
        break;
      }
      // the unit's sums over this CTA's steps: the four phases in order
      float v[kGvRows];
#pragma unroll
      for (int t = 0; t < kGvRows; ++t) {
        const float* src = red + ((rs * kGvPhases) * kGvRows + t) * kBM + tid;
        v[t] = ((src[0] + src[kGvRows * kBM]) + src[2 * kGvRows * kBM]) + src[3 * kGvRows * kBM];
      }
      // (the slot is released at the end of this unit's epilogue: the SwiGLU
      // stages the sums in its first phase's part, where each thread has just
      // read its own row)
      float* fin = red + (rs * kGvPhases * kGvRows) * kBM;
      ++ru;
      if (tid == 0) GV_STAMP(6);

      if (down) {
#pragma unroll
        for (int t = 0; t < kGvRows; ++t) {
          if (t >= T) break;
          const int slot = tl.slot[t];
          int e = D.rowexp[tl.p0 + t];
          e = e < -kMaxRowExp ? -kMaxRowExp : (e > kMaxRowExp ? kMaxRowExp : e);
          const float wt = D.topk_weights[slot] * exp2_int(2 * e);
          const long long ai = static_cast<long long>(slot / D.topk) * D.Kout + static_cast<long long>(rt) * kBM + tid;
          if (MOE_CHECK(ai >= 0 && ai < D.acc_elems, a.status, a.dbg, 43, ai, slot)) atomicAdd(D.acc + ai, wt * v[t]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kGbRedEmpty + rs));
        continue;
      }
      // gate/up: a unit cut between CTAs is finished by its last contributor
      bool write_tile = kb0 == 0 && kb1 == a.KBn;
      if (!write_tile) {
        const long long ustart = u * a.KBn;
        const int part = (my_begin < ustart) ? 1 : 0;
        float* slot = a.scratch + (static_cast<long long>(blockIdx.x) * 2 + part) * kBNMax * kBM;
#pragma unroll
        for (int t = 0; t < kGvRows; ++t)
          if (t < T && MOE_CHECK((slot - a.scratch) + t * kBM + tid < a.scratch_elems, a.status, a.dbg, 44,
                                 blockIdx.x, t))
            __stcg(slot + t * kBM + tid, v[t]);
        __threadfence();
        named_bar_sync(kGvEpiBar, kGvEpiThreads);
        const int c0 = cta_of(ustart), c1 = cta_of(ustart + a.KBn - 1);
        if (tid == 0) {
          const int add = kb1 - kb0;
          const int old = atomicAdd(a.tickets + c0, add);
          *last_flag = (old + add == a.KBn) ? 1 : 0;
        }
        named_bar_sync(kGvEpiBar, kGvEpiThreads);
        write_tile = *last_flag != 0;
        if (write_tile) {
          __threadfence();
#pragma unroll
          for (int t = 0; t < kGvRows; ++t) v[t] = 0.f;
          for (int cc = c0; cc <= c1; ++cc) {
            if (bounds[cc] == bounds[cc + 1]) continue;  // empty share: no partial
            const int pc = (bounds[cc] < ustart) ? 1 : 0;
            const float* sl = a.scratch + (static_cast<long long>(cc) * 2 + pc) * kBNMax * kBM;
#pragma unroll
            for (int t = 0; t < kGvRows; ++t)
              if (t < T) v[t] += __ldcg(sl + t * kBM + tid);
          }
        }
      }
      if (write_tile) {
        // h = SiLU(g) * u for the tile's 64 features: rows 2i (gate) and 2i + 1 (up)
#pragma unroll
        for (int t = 0; t < kGvRows; ++t) fin[t * kBM + tid] = v[t];
        named_bar_sync(kGvEpiBar, kGvEpiThreads);
        const int f = tid & 63;  // feature within the tile; a warp holds 32 of one token
        for (int t = tid >> 6; t < T; t += 2) {
          const int p = tl.p0 + t;
          const int e_raw = a.rowexp[p];
          const int e = e_raw < -kMaxRowExp ? -kMaxRowExp : (e_raw > kMaxRowExp ? kMaxRowExp : e_raw);
          const float sc_e = exp2_int(e);
          const float g = fin[t * kBM + 2 * f] * sc_e;
          const float uu = fin[t * kBM + 2 * f + 1] * sc_e;
          const float sig = __fdividef(1.0f, 1.0f + __expf(-g));
          float hv = g * sig * uu * exp2_int(-2 * e);
          sat = sat || fabsf(hv) > 65504.0f;
          hv = fminf(fmaxf(hv, -65504.0f), 65504.0f);
          const __half hh = __float2half_rn(hv);
          const long long hoff = (static_cast<long long>(rt) * a.Gcap + p / kRowGroup) * kRowGroupBytes +
                                 blocked_offset(p % kRowGroup, f);
          if (MOE_CHECK(hoff >= 0 && hoff + 2 <= a.hout_bytes, a.status, a.dbg, 45, hoff, p))
            *reinterpret_cast<__half*>(a.hout + hoff) = hh;
          // h as a step row of the down product (its step rt / 2 holds this
          // tile's 64 features at (rt % 2) * 64): this warp's 32 features are one
          // scale group of it, in 16-bit block fixed point (layout.cuh)
          uint8_t* xs = a.xv_out + (static_cast<long long>(tl.slot[t]) * (a.R / 2) + (rt >> 1)) * kXvStepBytes;
          const bool xs_ok = MOE_CHECK((xs - a.xv_out) + kXvStepBytes <= a.xv_out_bytes, a.status, a.dbg, 46,
                                       xs - a.xv_out, p);
          float m = fabsf(hv);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          const int eg = xv_group_exp(m);
          const int v16 = xv_quantize(hv, eg);
          int sum = v16;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          const int gi = 2 * (rt & 1) + (f >> 5);
          if (xs_ok) {
            *reinterpret_cast<int16_t*>(xs + gi * 64 + ((f & 31) >> 3) * 16 + xv_slot(f & 7) * 2) =
                static_cast<int16_t>(v16);
            if (lane == 0) xv_header(xs, gi, sum, eg);
          }
        }
        if (kMode == 3) __threadfence();  // (the step rows are read by other CTAs' copiers)
        named_bar_sync(kGvEpiBar, kGvEpiThreads);  // every thread is done with the staged sums
        // one launch: the second of the two row tiles of the down step rt / 2 makes
        // its rows ready
        if (kMode == 3 && tid == 0) atomicAdd(b.h_ready + (u / R) * b.KBn + (rt >> 1), 1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kGbRedEmpty + rs));
    }
    }
    if (__any_sync(0xffffffffu, sat) && lane == 0) atomicOr(status, kStatusHSaturated);
  }

  // ------------------------------------------------ teardown
  // Every copy issued is waited for by its readers unless a wait gave up. Then
  // thread 0 lets the latest copy into every slot land before it exits (the
  // CTA's shared memory lives until its last thread has exited).
  __syncwarp();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag != 0) {
    for (int i = 0; i < kGvNWS; ++i)
      if (wlast[i] >= 0) mbar_wait_drain(bar(kGbWFull + i), static_cast<uint32_t>((wlast[i] / kGvNWS) & 1));
    for (int i = 0; i < kGvNB; ++i)
      if (blast[i] >= 0) mbar_wait_drain(bar(kGbBFull + i), static_cast<uint32_t>((blast[i] / kGvNB) & 1));
  }
  if (threadIdx.x == 0) GV_STAMP(7);
}

}  // namespace

static cudaError_t launch_gemv(void (*kernel)(GemmArgs, GemmArgs), const GemmArgs& a, int num_ctas,
                               cudaStream_t stream, bool pdl) {
  return launch_k(kernel, dim3(static_cast<unsigned>(num_ctas)), dim3(kGvThreads), kGsAlloc, stream, pdl, a, a);
}
cudaError_t launch_gemv_gateup(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_gemv(gemv_kernel<1>, a, num_ctas, stream, pdl);
}
cudaError_t launch_gemv_down(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_gemv(gemv_kernel<2>, a, num_ctas, stream, pdl);
}
cudaError_t launch_gemv_both(const GemmArgs& a1, const GemmArgs& a2, int num_ctas, cudaStream_t stream, bool pdl) {
  return launch_k_coop(gemv_kernel<3>, dim3(static_cast<unsigned>(num_ctas)), dim3(kGvThreads), kGsAlloc, stream,
                       pdl, a1, a2);
}
cudaError_t gemv_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGsAlloc);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGsAlloc);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGsAlloc);
  return e;
}

}  // namespace moe
