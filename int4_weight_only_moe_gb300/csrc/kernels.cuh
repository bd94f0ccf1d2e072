// Launchers of the forward's kernels (each defined in its own translation unit).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "layout.cuh"
#include "ptx.cuh"

namespace moe {

// Sets *bad_scale (device) when a scale lies outside the supported range.
// Source layouts of the repack (see pack.cu).
constexpr int kLayoutGptq = 0;
constexpr int kLayoutCompressedTensors = 1;
struct RepackSource {
  const int32_t* q;         // codes (null for the unpack direction)
  const uint16_t* s;        // bf16 scales
  int layout;               // kLayoutGptq or kLayoutCompressedTensors
  const int32_t* red_perm;  // [E, Kred] packed -> source reduction element (act-order), or null
  const int32_t* out_perm;  // [E, out_period] packed -> source output feature, or null
  int out_period;
  int Kred, Nout;
};
cudaError_t launch_repack(const RepackSource& src, uint8_t* out, int E, int R, int KBn,
                          int interleave, int32_t* bad_scale, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* in, const RepackSource& dst, int32_t* q, uint16_t* s, int E,
                          int R, int KBn, int interleave, cudaStream_t stream);
// Act-order packing order [E, R] from the group index [E, R]; *bad set on an
// index out of range or a group without exactly 32 elements.
cudaError_t launch_perm_from_g_idx(const int32_t* g_idx, int32_t* perm, int E, int R, int32_t* bad,
                                   cudaStream_t stream);

// Token->expert align (counting sort + padding + token-tile list). With bn_max == 0
// no tile list is written (the debug entry point); expert_offsets may be null.
struct AlignArgs {
  const int32_t* topk_ids;  // device, or the routing kernel's own shared-memory copy
  // small-batch launch only: route the tokens' router logits [M, E] here first
  // (null: topk_ids are given), writing ids and weights to ids_out / wts_out
  const float* logits;
  int32_t* ids_out;
  float* wts_out;
  int M_tokens, topk;
  int MK;             // M * topk (flat slot count; also the padding sentinel)
  int E;              // experts held (local experts under expert parallelism)
  int e_begin, E_total;  // the held experts are [e_begin, e_begin + E) of E_total
  int block;          // per-expert padding granularity
  int bn_max;         // token-tile size (multiple of 16) or 0
  int32_t* sorted_ids;
  int32_t* expert_offsets;  // [E + 1] or null
  TokenTile* tiles;         // or null
  int32_t* expert_tiles;    // [E] token tiles per expert, or null
  int32_t* hdr;             // workspace header (status, num_padded, num_tiles)
  int32_t* tickets;         // zeroed, or null
  int n_tickets;            // (tickets holds n_tickets entries, all zeroed)
  int32_t* num_padded_out;  // optional extra copy of num_padded
  int sorted_cap, tiles_cap;  // extents for the self-checking build
  int32_t* dbg;
  // cost-weighted stream-K boundaries (general path; null: not computed):
  // sched[w * (sched_ctas + 1) + c] = first step of CTA c in GEMM w (0 gate/up,
  // 1 down), whose units are (row tiles sched_R[w]) x (steps sched_KBn[w])
  long long* sched;
  int sched_ctas;
  int sched_R[2], sched_KBn[2];
  int step_cost_per_group[2];  // per GEMM; 0 = even split for that GEMM
  // the CUDA-core products' tile list (every expert's rows in tiles of at most
  // kGemvRows, experts in id order; count in hdr[kHdrNumGemvTiles]), or null
  GemvTile* gv_tiles;
  int gv_tiles_cap;
};
cudaError_t launch_align(const AlignArgs& a, cudaStream_t stream, bool pdl);
// At handle creation: the general align kernel's dynamic shared memory limit,
// sized for the largest expert count.
cudaError_t align_set_attributes(int E);

// Expert-sorted, blocked copy of the hidden states; also zeroes the fp32 accumulator.
struct GatherArgs {
  const uint16_t* x;  // [M, K] bf16
  const int32_t* sorted_ids;
  const int32_t* hdr;
  int MK, topk, K, Gcap;
  uint8_t* xs;        // blocked [K/64][Gcap][16 x 128 B]
  int32_t* rowexp;    // [padded rows] prescale exponent of each expert-sorted row
  float* acc;         // [M, K] fp32, zeroed
  long long acc_elems;
  long long xs_bytes;  // extents for the self-checking build
  int M;
  int32_t* dbg;
  // act-order on w1: packed reduction element j of expert e is hidden element
  // perm1[e][j]; the gather writes the row in that order (null: natural order)
  const int32_t* perm1;
  const int32_t* topk_ids;  // expert of a slot (read only when perm1 is set)
  int e_begin;              // first expert held (the ids are the layer's)
  // small-batch CUDA-core path: write the rows as step rows (layout.cuh, with
  // xv_steps = K / 128 steps a row) instead of the blocked layout (null: blocked)
  uint8_t* xv;
  int xv_steps;
};
cudaError_t launch_gather(const GatherArgs& a, int max_groups, int num_sms, cudaStream_t stream,
                          bool pdl);
// M * topk <= 32: the routing (as the align kernel) and the gather in one launch.
// max_rows bounds the padded rows (the workspace's capacity).
cudaError_t launch_route_gather_small(const AlignArgs& a, const GatherArgs& g, int max_rows,
                                      int num_sms, cudaStream_t stream, bool pdl);

// Router: top-k routing of logits [M, E] into ids / weights [M, k] (k <= 32).
cudaError_t launch_route(const float* logits, int M, int E, int k, int32_t* ids, float* wts,
                         int num_sms, cudaStream_t stream, bool pdl);

// The fused small-batch launch's own preparation (what the routing + gather
// kernel does otherwise) and its cross-CTA counters, kept in the handle: fsync
// holds [kFsStatus] the status word, [kFsPrep] CTAs done preparing, [kFsExit]
// CTAs done, then the split-unit tickets, K/128 reserved words and the
// intermediate counters; all zero between calls (the last CTA to finish clears
// them). The workspace header receives the status and the row counts at the end.
enum { kFsStatus = 0, kFsPrep = 1, kFsExit = 2, kFsTickets = 8 };
struct FusedPrep {
  const uint16_t* x;         // hidden bf16 [M, K]
  uint8_t* xs;               // blocked B operand of the gate/up GEMM
  int32_t* sorted_ids;       // [padded rows] flat slot of each expert-sorted row
  int32_t* rowexp;           // [padded rows] prescale exponent
  float* acc;                // [M, K] fp32 output accumulator, zeroed here
  long long acc_elems;
  const int32_t* perm1;      // act-order packing order of w1 [E, K], or null
  int32_t* fsync;            // handle's counters (see above)
  int fsync_words;
  int32_t* ws_hdr;           // workspace header
  int K, topk;
};

struct GemmArgs {
  const uint8_t* wpack;    // packed weights of this GEMM
  const uint8_t* bsrc;     // blocked activations (B operand)
  const int32_t* hdr;
  const TokenTile* tiles;
  const int32_t* expert_tiles;
  const int32_t* rowexp;   // prescale exponent of each expert-sorted row
  // at most 32 routed slots: the caller's topk_ids [MK], from which the kernel
  // recomputes the routing tiles itself (so its weight stream need not wait for
  // the preceding kernel); null: read the tiles the align kernel wrote
  const int32_t* small_ids;
  int e_begin, E_total;    // the held experts are [e_begin, e_begin + E) of E_total (small_ids)
  uint32_t wait_kcycles;   // pipeline wait limit in units of 1024 SM cycles (wait_limit_kcycles)
  int test_never_wait;     // test hook: the epilogue first waits on a barrier nothing arrives on
  // fused small-batch launch: per token tile and down-GEMM k-block, a zeroed
  // counter of the gate/up row tiles whose intermediate is stored ([32][N/128])
  int32_t* h_ready;
  FusedPrep prep;          // fused launch only
  int R;                   // row tiles per expert
  int KBn;                 // k-blocks per unit
  int Gcap;                // row groups per k-block plane of bsrc / hout
  // gate/up GEMM
  uint8_t* hout;           // blocked intermediate activations [N/64][Gcap][...]
  float* scratch;          // split-K partial tiles [kMaxCtas][2][kBNMax][128]
  int32_t* tickets;        // [kMaxCtas]
  // down GEMM
  const int32_t* sorted_ids;
  const float* topk_weights;
  float* acc;              // [M, Kout] fp32
  int Kout, MK, topk;
  int32_t* status;
  // buffer extents, read only by the self-checking build (-DMOE_CHECKS)
  long long wpack_bytes, bsrc_bytes, hout_bytes, acc_elems, scratch_elems;
  int sorted_cap, tiles_cap, E;
  int32_t* dbg;  // first failed check: site, values, block, thread
  const long long* sched;  // [gridDim.x + 1] weighted boundaries, used when this GEMM's
                           // bit of hdr[kHdrSched] is set (bit 0 gate/up, bit 1 down)
  // small-batch CUDA-core kernels: the activation rows as step rows (xv_in; the
  // gate/up kernel also writes h as step rows of the down product, xv_out)
  const uint8_t* xv_in;
  uint8_t* xv_out;
  long long xv_bytes, xv_out_bytes;
  // more than 32 routed slots: the align kernel's CUDA-core tile list (small_ids null)
  const GemvTile* gv_tiles;
  int Pcap;
  int ids_after_pdl;       // small_ids is the preceding kernel's output (routed in-launch)
};
cudaError_t launch_gemm_gateup(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl);
cudaError_t launch_gemm_down(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl);
// Both GEMMs in one cooperative launch (small batches: small_ids set in both).
cudaError_t launch_gemm_fused(const GemmArgs& a1, const GemmArgs& a2, int num_ctas, cudaStream_t stream,
                              bool pdl);
cudaError_t gemm_set_attributes();
// The same two products for a batch of at most 32 routed slots on the CUDA cores
// (small_ids set; xv_in / xv_out set): tiles of at most 4 token rows per expert.
cudaError_t launch_gemv_gateup(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl);
cudaError_t launch_gemv_down(const GemmArgs& a, int num_ctas, cudaStream_t stream, bool pdl);
// both CUDA-core products of a batch of at most 32 routed slots in one cooperative launch
cudaError_t launch_gemv_both(const GemmArgs& a1, const GemmArgs& a2, int num_ctas, cudaStream_t stream, bool pdl);
cudaError_t gemv_set_attributes();

cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            cudaStream_t stream, bool pdl);

cudaError_t launch_read_intermediate(const uint8_t* hbuf, const int32_t* sorted_ids,
                                     const int32_t* rowexp, const int32_t* hdr, int MK, int N,
                                     int Gcap, int max_rows, float* h_rows, cudaStream_t stream);

// Self-checking build (-DMOE_CHECKS): every global access is range-checked first;
// a failed check sets status bit 8, records the first failure (site, two values,
// block, thread) in dbg[0..5] and skips the access.
#ifdef MOE_CHECKS
__device__ __forceinline__ bool moe_check(bool ok, int32_t* status, int32_t* dbg, int site,
                                          long long v0, long long v1) {
  if (!ok) {
    if (status) atomicOr(status, 8);
    if (dbg && atomicCAS(dbg, 0, site) == 0) {
      dbg[1] = static_cast<int32_t>(v0);
      dbg[2] = static_cast<int32_t>(v1);
      dbg[3] = static_cast<int32_t>(blockIdx.x);
      dbg[4] = static_cast<int32_t>(threadIdx.x);
      dbg[5] = static_cast<int32_t>(v0 >> 32);
    }
  }
  return ok;
}
#define MOE_CHECK(cond, status, dbg, site, v0, v1) \
  moe_check((cond), (status), (dbg), (site), (long long)(v0), (long long)(v1))
#else
#define MOE_CHECK(cond, status, dbg, site, v0, v1) true
#endif

// Launch helper: optional programmatic dependent launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// The same as a cooperative launch: every CTA of the grid is resident at once
// (or the launch fails), as kernels whose CTAs wait on one another need.
template <typename... KArgs, typename... Args>
cudaError_t launch_k_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
