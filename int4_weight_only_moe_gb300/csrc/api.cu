// C-ABI of the W4A16 fused MoE library: handle, argument checks, workspace
// layout and the launch sequence of the forward
//   align -> gather -> gate/up GEMM -> down GEMM -> finalize.
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/moe_w4a16.h"
#include "kernels.cuh"

using namespace moe;

struct moe_w4a16_ctx {
  int E, K, N, topk, group;
  int e_begin, E_total;  // expert parallelism: the handle holds [e_begin, e_begin + E) of E_total
  int device;
  int num_sms;
  int num_ctas;
  int step_cost[2];  // per GEMM (gate/up, down): stream-K cost per row group beyond two (0: even split)
  bool pdl;
  bool profile;
  unsigned long long wait_us;  // GEMM pipeline wait limit (0: the kernels' default)
  bool test_never_wait;        // test hook (MOE_W4A16_OPT_TEST_WAIT_NEVER_COMPLETES)
  bool fused_small;            // MOE_W4A16_OPT_FUSED_SMALL_BATCH
  int gemv_small;              // MOE_W4A16_OPT_GEMV_SMALL_BATCH (0, 1 and 3: <= 256 slots, 2: one token)
  bool gemv_one_launch;        // MOE_W4A16_OPT_GEMV_ONE_LAUNCH
  int32_t* dflag;              // device words: pack's scale check [0], g_idx check [1]
  uint8_t* w1p;
  uint8_t* w2p;
  size_t w1p_bytes, w2p_bytes;
  bool packed;
  int layout;      // source layout of the last pack (for the inverse)
  int32_t* perm1;  // act-order packing order of w1's reduction elements [E, K], or null
  int32_t* perm2;  // the same for w2 [E, N] (also the order of w1's output features)
  int32_t* fsync;  // the fused small-batch launch's counters (zero between calls)
  int fsync_words;
  cudaEvent_t ev[6];
  bool ev_valid;
  // pinned staging of small host-buffer forwards whose buffers are pageable
  uint8_t* hstage;
  size_t hstage_bytes;
};

namespace {

thread_local std::string g_last_error = "no error";

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

#define MOE_CUDA_TRY(expr)                                                                   \
  do {                                                                                       \
    cudaError_t e_ = (expr);                                                                 \
    if (e_ != cudaSuccess)                                                                   \
      return fail(MOE_W4A16_CUDA_ERROR, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Host-buffer forwards whose hidden states are at most this large let the kernels
// read the inputs and write the output in host memory over the host-device link
// (zero-copy); larger ones move them with the copy engines, which stream large
// transfers faster than the gather and finalize kernels' loads and stores would.
constexpr size_t kZeroCopyMaxBytes = 1u << 20;

// Default stream-K cost of a pipeline step per row group of its token tile beyond
// the second, in eighths of a one-group step, per GEMM. Measured on GB300 with
// Zipf-routed M = 1024 (hot experts in full 64-row tiles): weighting the down
// GEMM by 2 took the forward from 2,923 to 2,653 us; weighting the gate/up GEMM,
// or the down GEMM by more, was slower; other batch sizes do not change.
constexpr int kDefaultStepCostGateUp = 0;
constexpr int kDefaultStepCostDown = 2;

// Device address of a pinned (page-locked or registered) host buffer, or null if
// `p` is pageable memory the device cannot address.
const void* pinned_device_pointer(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

struct WsLayout {
  size_t hdr, tickets, sched, sorted, rowexp, tiles, expert_tiles, xs, hbuf, scratch, acc, xv1, xv2, gv_tiles,
      total;
  int Pcap, Gcap;
};

// Workspace carve-up for M tokens. Pcap bounds the padded routed-row count:
// M*k rows plus at most 15 padding rows for each expert that receives any.
int n_tickets(const moe_w4a16_ctx* h) { return kMaxCtas + h->K / kBM + kSmallTiles * (h->N / kBM); }

WsLayout ws_layout(const moe_w4a16_ctx* h, int M) {
  WsLayout L{};
  const long long MK = static_cast<long long>(M) * h->topk;
  const long long active = MK < h->E ? MK : h->E;
  long long pcap = align_up(static_cast<size_t>(MK + active * (kRowGroup - 1)), kRowGroup);
  if (pcap < kRowGroup) pcap = kRowGroup;
  L.Pcap = static_cast<int>(pcap);
  L.Gcap = L.Pcap / kRowGroup;
  size_t off = 0;
  L.hdr = off;
  off += kHdrWords * sizeof(int32_t);
  off = align_up(off, 256);
  // gate/up split-unit tickets [kMaxCtas], the down row-tile tickets [K/128], then
  // the fused launch's intermediate counters [32 token tiles][N/128]
  L.tickets = off;
  off = align_up(off + n_tickets(h) * sizeof(int32_t), 256);
  L.sched = off;  // stream-K boundaries of the two GEMMs
  off = align_up(off + 2 * (kMaxCtas + 1) * sizeof(long long), 256);
  L.sorted = off;
  off = align_up(off + static_cast<size_t>(L.Pcap) * sizeof(int32_t), 256);
  L.rowexp = off;
  off = align_up(off + static_cast<size_t>(L.Pcap) * sizeof(int32_t), 256);
  L.tiles = off;
  off = align_up(off + static_cast<size_t>(L.Gcap) * sizeof(TokenTile), 256);
  L.expert_tiles = off;
  off = align_up(off + static_cast<size_t>(h->E) * sizeof(int32_t), 1024);
  // (the blocked hidden rows, or for the CUDA-core products their step rows)
  // (sized for min(M * topk, kGemvMaxSlots) rows whatever the path, so that the
  // size never shrinks as M grows)
  const size_t xv_rows = static_cast<size_t>(MK < kGemvMaxSlots ? MK : kGemvMaxSlots);
  L.xs = off;
  const size_t xs_blocked = static_cast<size_t>(L.Pcap) * h->K * 2;
  const size_t xs_rows = xv_rows * (h->K / 128) * kXvStepBytes;
  off = align_up(off + (xs_blocked > xs_rows ? xs_blocked : xs_rows), 1024);
  L.hbuf = off;
  off = align_up(off + static_cast<size_t>(L.Pcap) * h->N * 2, 1024);
  L.scratch = off;  // (a pair of split-unit slots per CTA of the handle's grid)
  off = align_up(off + static_cast<size_t>(h->num_ctas) * 2 * kBNMax * kBM * sizeof(float), 1024);
  L.acc = off;
  off = align_up(off + static_cast<size_t>(M) * h->K * sizeof(float), 1024);
  // batches the CUDA-core products can take (at most kGemvMaxSlots routed slots):
  // the gathered hidden rows as step rows (layout.cuh; one row per routed slot, in
  // the region of the blocked rows, which those products do not read), the
  // intermediate as step rows, and the tile list
  L.xv1 = L.xs;
  L.xv2 = off;
  off = align_up(off + xv_rows * (h->N / 128) * kXvStepBytes, 1024);
  L.gv_tiles = off;
  off = align_up(off + xv_rows * sizeof(GemvTile), 1024);
  L.total = off;
  return L;
}

size_t staging_bytes(const moe_w4a16_ctx* h, int M) {
  const size_t mk = static_cast<size_t>(M) * h->topk;
  return align_up(static_cast<size_t>(M) * h->K * 2, 256) * 2 + align_up(mk * 4, 256) * 2;
}

int check_handle(const moe_w4a16_ctx* h) {
  if (!h) return fail(MOE_W4A16_INVALID_ARG, "null handle");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device)
    return fail(MOE_W4A16_INVALID_ARG, "current CUDA device differs from the handle's device");
  return MOE_W4A16_OK;
}

}  // namespace

namespace moe {
// Record `msg` as this thread's last error and return `code` (for entry points
// defined in other translation units).
int report_error(int code, const char* msg) { return fail(code, msg); }
}  // namespace moe

extern "C" {

const char* moe_w4a16_last_error(void) { return g_last_error.c_str(); }

int moe_w4a16_create(int E, int K, int N, int topk, int group_size, moe_w4a16_t* out) {
  if (!out) return fail(MOE_W4A16_INVALID_ARG, "out is null");
  *out = nullptr;
  if (group_size != kGroup) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "group_size must be 32");
  if (E < 1 || E > kMaxExperts) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "E must be in [1, 1024]");
  if (topk < 1 || topk > E) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "topk must be in [1, E]");
  if (K <= 0 || K % 128 != 0) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "K must be a positive multiple of 128");
  if (N <= 0 || N % 128 != 0) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "N must be a positive multiple of 128");
  auto* h = new moe_w4a16_ctx();
  std::memset(h, 0, sizeof(*h));
  h->E = E;
  h->E_total = E;
  h->K = K;
  h->N = N;
  h->topk = topk;
  h->group = group_size;
  h->pdl = true;
  h->fused_small = false;
  h->gemv_small = 1;
  h->gemv_one_launch = false;
  h->step_cost[0] = kDefaultStepCostGateUp;
  h->step_cost[1] = kDefaultStepCostDown;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess) e = gemm_set_attributes();
  if (e == cudaSuccess) e = gemv_set_attributes();
  if (e == cudaSuccess) e = align_set_attributes(E);
  if (e != cudaSuccess) {
    delete h;
    return fail(MOE_W4A16_CUDA_ERROR, std::string("device setup: ") + cudaGetErrorString(e));
  }
  h->num_ctas = h->num_sms < kMaxCtas ? h->num_sms : kMaxCtas;
  // w1: 2N rows x K, w2: K rows x N; half a byte per code plus 2 bytes per 32 codes
  h->w1p_bytes = static_cast<size_t>(E) * (2 * N / kBM) * (K / kBK) * kWBlockBytes;
  h->w2p_bytes = static_cast<size_t>(E) * (K / kBM) * (N / kBK) * kWBlockBytes;
  e = cudaMalloc(&h->w1p, h->w1p_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->w2p, h->w2p_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&h->dflag, 256);
  h->fsync_words = kFsTickets + kMaxCtas + K / kBM + kSmallTiles * (N / kBM);
  if (e == cudaSuccess) e = cudaMalloc(&h->fsync, static_cast<size_t>(h->fsync_words) * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->fsync, 0, static_cast<size_t>(h->fsync_words) * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->w1p);
    cudaFree(h->w2p);
    delete h;
    return fail(MOE_W4A16_CUDA_ERROR, std::string("cudaMalloc packed weights: ") + cudaGetErrorString(e));
  }
  *out = h;
  return MOE_W4A16_OK;
}

int moe_w4a16_create_ep(int E_total, int expert_begin, int expert_end, int K, int N, int topk,
                        int group_size, moe_w4a16_t* out) {
  if (!out) return fail(MOE_W4A16_INVALID_ARG, "out is null");
  *out = nullptr;
  if (E_total < 1 || E_total > kMaxExperts)
    return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "E_total must be in [1, 1024]");
  if (expert_begin < 0 || expert_end <= expert_begin || expert_end > E_total)
    return fail(MOE_W4A16_INVALID_ARG, "need 0 <= expert_begin < expert_end <= E_total");
  if (topk < 1 || topk > E_total) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "topk must be in [1, E_total]");
  const int E = expert_end - expert_begin;
  // (the local handle may hold fewer experts than a token's top-k)
  int rc = moe_w4a16_create(E, K, N, topk <= E ? topk : E, group_size, out);
  if (rc != MOE_W4A16_OK) return rc;
  (*out)->topk = topk;
  (*out)->e_begin = expert_begin;
  (*out)->E_total = E_total;
  return MOE_W4A16_OK;
}

int moe_w4a16_destroy(moe_w4a16_t h) {
  if (!h) return fail(MOE_W4A16_INVALID_ARG, "null handle");
  cudaDeviceSynchronize();
  cudaFree(h->w1p);
  cudaFree(h->w2p);
  cudaFree(h->dflag);
  cudaFree(h->fsync);
  cudaFree(h->perm1);
  cudaFree(h->perm2);
  if (h->hstage) cudaFreeHost(h->hstage);
  if (h->ev_valid)
    for (auto& ev : h->ev) cudaEventDestroy(ev);
  delete h;
  return MOE_W4A16_OK;
}

size_t moe_w4a16_packed_bytes(moe_w4a16_t h) { return h ? h->w1p_bytes + h->w2p_bytes : 0; }

int moe_w4a16_pack(moe_w4a16_t h, const int32_t* w1_q, const uint16_t* w1_s, const int32_t* w2_q,
                   const uint16_t* w2_s, void* stream) {
  return moe_w4a16_pack_ex(h, w1_q, w1_s, w2_q, w2_s, MOE_W4A16_LAYOUT_GPTQ, nullptr, nullptr, stream);
}

namespace {

// Source description of w1 (gate/up: reduction K, 2N output features, features
// reordered by w2's act-order permutation) and of w2 (reduction N, K features).
RepackSource w1_source(moe_w4a16_t h, const int32_t* q, const uint16_t* sc) {
  return RepackSource{q, sc, h->layout, h->perm1, h->perm2, h->N, h->K, 2 * h->N};
}
RepackSource w2_source(moe_w4a16_t h, const int32_t* q, const uint16_t* sc) {
  return RepackSource{q, sc, h->layout, h->perm2, nullptr, 0, h->N, h->K};
}

// Act-order packing order of one matrix from its group index, or none.
int make_perm(moe_w4a16_t h, const int32_t* g_idx, int R, int32_t** perm, cudaStream_t s) {
  cudaFree(*perm);
  *perm = nullptr;
  if (!g_idx) return MOE_W4A16_OK;
  MOE_CUDA_TRY(cudaMalloc(perm, static_cast<size_t>(h->E) * R * sizeof(int32_t)));
  MOE_CUDA_TRY(launch_perm_from_g_idx(g_idx, *perm, h->E, R, h->dflag + 1, s));
  return MOE_W4A16_OK;
}

}  // namespace

int moe_w4a16_pack_ex(moe_w4a16_t h, const int32_t* w1_q, const uint16_t* w1_s, const int32_t* w2_q,
                      const uint16_t* w2_s, int layout, const int32_t* w1_g_idx,
                      const int32_t* w2_g_idx, void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!w1_q || !w1_s || !w2_q || !w2_s) return fail(MOE_W4A16_INVALID_ARG, "null weight pointer");
  if (layout != MOE_W4A16_LAYOUT_GPTQ && layout != MOE_W4A16_LAYOUT_COMPRESSED_TENSORS)
    return fail(MOE_W4A16_INVALID_ARG, "unknown weight layout");
  auto s = static_cast<cudaStream_t>(stream);
  h->packed = false;
  h->layout = layout == MOE_W4A16_LAYOUT_GPTQ ? kLayoutGptq : kLayoutCompressedTensors;
  MOE_CUDA_TRY(cudaMemsetAsync(h->dflag, 0, 2 * sizeof(int32_t), s));
  if (int rc = make_perm(h, w1_g_idx, h->K, &h->perm1, s)) return rc;
  if (int rc = make_perm(h, w2_g_idx, h->N, &h->perm2, s)) return rc;
  int32_t flags[2] = {0, 0};
  if (h->perm1 || h->perm2) {  // a bad group index stops here, before any repack reads it
    MOE_CUDA_TRY(cudaMemcpyAsync(flags, h->dflag, sizeof(flags), cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    if (flags[1])
      return fail(MOE_W4A16_BAD_G_IDX,
                  "g_idx: every group index must lie in [0, R/32) and every group hold exactly 32 "
                  "elements");
  }
  MOE_CUDA_TRY(launch_repack(w1_source(h, w1_q, w1_s), h->w1p, h->E, 2 * h->N / kBM, h->K / kBK, 1,
                             h->dflag, s));
  MOE_CUDA_TRY(launch_repack(w2_source(h, w2_q, w2_s), h->w2p, h->E, h->K / kBM, h->N / kBK, 0,
                             h->dflag, s));
  MOE_CUDA_TRY(cudaMemcpyAsync(flags, h->dflag, sizeof(flags), cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  if (flags[0])
    return fail(MOE_W4A16_UNSUPPORTED_SCALE,
                "a scale is outside the supported range (0, or 2^-14 <= |s| <= 2720, finite): "
                "its fp16 dequantised weights would not be exact");
  h->packed = true;
  return MOE_W4A16_OK;
}

int moe_w4a16_unpack_debug(moe_w4a16_t h, int32_t* w1_q, uint16_t* w1_s, int32_t* w2_q,
                           uint16_t* w2_s, void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!w1_q || !w1_s || !w2_q || !w2_s) return fail(MOE_W4A16_INVALID_ARG, "null weight pointer");
  if (!h->packed) return fail(MOE_W4A16_NOT_PACKED, "weights not packed");
  auto s = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(launch_unpack(h->w1p, w1_source(h, nullptr, nullptr), w1_q, w1_s, h->E, 2 * h->N / kBM,
                             h->K / kBK, 1, s));
  MOE_CUDA_TRY(launch_unpack(h->w2p, w2_source(h, nullptr, nullptr), w2_q, w2_s, h->E, h->K / kBM,
                             h->N / kBK, 0, s));
  return MOE_W4A16_OK;
}

size_t moe_w4a16_workspace_size(moe_w4a16_t h, int M) {
  if (!h || M < 0) return 0;
  return ws_layout(h, M).total;
}

size_t moe_w4a16_host_staging_size(moe_w4a16_t h, int M) {
  if (!h || M < 0) return 0;
  return staging_bytes(h, M);
}

int moe_w4a16_set_option(moe_w4a16_t h, int option, int value) {
  if (!h) return fail(MOE_W4A16_INVALID_ARG, "null handle");
  switch (option) {
    case MOE_W4A16_OPT_NUM_CTAS:
      if (value < 1 || value > kMaxCtas) return fail(MOE_W4A16_INVALID_ARG, "num_ctas must be in [1, 256]");
      h->num_ctas = value;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_PROFILE:
      if (value && !h->ev_valid) {
        for (auto& ev : h->ev) MOE_CUDA_TRY(cudaEventCreate(&ev));
        h->ev_valid = true;
      }
      h->profile = value != 0;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_PDL:
      h->pdl = value != 0;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_WAIT_LIMIT_US:
      if (value < 0) return fail(MOE_W4A16_INVALID_ARG, "wait limit must be >= 0");
      h->wait_us = static_cast<unsigned long long>(value);
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_FUSED_SMALL_BATCH:
      h->fused_small = value != 0;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_GEMV_SMALL_BATCH:
      if (value < 0 || value > 3) return fail(MOE_W4A16_INVALID_ARG, "GEMV option must be 0, 1, 2 or 3");
      h->gemv_small = value;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_GEMV_ONE_LAUNCH:
      h->gemv_one_launch = value != 0;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_TEST_WAIT_NEVER_COMPLETES:
      h->test_never_wait = value != 0;
      return MOE_W4A16_OK;
    case MOE_W4A16_OPT_STEP_COST_GATEUP:
    case MOE_W4A16_OPT_STEP_COST_DOWN:
      if (value < 0 || value > 64) return fail(MOE_W4A16_INVALID_ARG, "step cost must be in [0, 64]");
      h->step_cost[option == MOE_W4A16_OPT_STEP_COST_DOWN ? 1 : 0] = value;
      return MOE_W4A16_OK;
    default:
      return fail(MOE_W4A16_INVALID_ARG, "unknown option");
  }
}

int moe_w4a16_kernel_times(moe_w4a16_t h, float* ms, int n) {
  if (!h || !ms) return fail(MOE_W4A16_INVALID_ARG, "null argument");
  if (!h->ev_valid) return fail(MOE_W4A16_INVALID_ARG, "profiling was never enabled");
  MOE_CUDA_TRY(cudaEventSynchronize(h->ev[5]));
  int w = 0;
  for (int i = 0; i < 5 && w < n; ++i, ++w) MOE_CUDA_TRY(cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]));
  return w;
}

}  // extern "C"

namespace {

// The forward's launch sequence. With `logits` the top-k routing runs first and
// writes topk_ids / topk_weights (outputs then); without, they are inputs.
int forward_impl(moe_w4a16_t h, const uint16_t* hidden, const float* logits, const int32_t* topk_ids,
                 const float* topk_weights, uint16_t* out, int M, void* workspace,
                 size_t workspace_bytes, void* stream, float* partial = nullptr) {
  if (int rc = check_handle(h)) return rc;
  if (M < 0) return fail(MOE_W4A16_INVALID_ARG, "M must be >= 0");
  if (M == 0) return MOE_W4A16_OK;
  if (!hidden || !topk_ids || !topk_weights || (!out && !partial) || !workspace)
    return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  if (partial && reinterpret_cast<uintptr_t>(partial) % 16 != 0)
    return fail(MOE_W4A16_INVALID_ARG, "partial must be 16-byte aligned");
  if (logits && h->topk > 32)
    return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "the router supports topk <= 32");
  if (!h->packed) return fail(MOE_W4A16_NOT_PACKED, "moe_w4a16_pack has not been called");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(MOE_W4A16_INVALID_ARG, "workspace must be 256-byte aligned");
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
    return fail(MOE_W4A16_INVALID_ARG, "hidden and out must be 16-byte aligned");
  const long long MK = static_cast<long long>(M) * h->topk;
  if (MK > (1LL << 26)) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "M * topk too large");
  const WsLayout L = ws_layout(h, M);
  if (workspace_bytes < L.total)
    return fail(MOE_W4A16_WORKSPACE_TOO_SMALL,
                "workspace too small: need " + std::to_string(L.total) + " bytes");
  auto s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  int32_t* tickets = reinterpret_cast<int32_t*>(ws + L.tickets);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  int32_t* rowexp = reinterpret_cast<int32_t*>(ws + L.rowexp);
  TokenTile* tiles = reinterpret_cast<TokenTile*>(ws + L.tiles);
  int32_t* expert_tiles = reinterpret_cast<int32_t*>(ws + L.expert_tiles);
  uint8_t* xs = ws + L.xs;
  uint8_t* hbuf = ws + L.hbuf;
  float* scratch = reinterpret_cast<float*>(ws + L.scratch);
  // (the partial-sum forward accumulates straight into the caller's buffer)
  float* acc = partial ? partial : reinterpret_cast<float*>(ws + L.acc);
  const bool prof = h->profile && h->ev_valid;
  const bool pdl = h->pdl && !prof;

  if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[0], s));
  AlignArgs aa{};
  aa.topk_ids = topk_ids;
  aa.M_tokens = M;
  aa.topk = h->topk;
  if (logits && MK <= 32) {  // routed inside the small-batch routing + gather launch
    aa.logits = logits;
    aa.ids_out = const_cast<int32_t*>(topk_ids);
    aa.wts_out = const_cast<float*>(topk_weights);
  }
  aa.MK = static_cast<int>(MK);
  aa.E = h->E;
  aa.e_begin = h->e_begin;
  aa.E_total = h->E_total;
  aa.block = kRowGroup;
  aa.bn_max = kBNMax;
  aa.sorted_ids = sorted;
  aa.tiles = tiles;
  aa.expert_tiles = expert_tiles;
  aa.hdr = hdr;
  aa.tickets = tickets;
  aa.n_tickets = n_tickets(h);
  aa.sorted_cap = L.Pcap;
  aa.tiles_cap = L.Gcap;
  aa.dbg = hdr + 8;
  // weighted stream-K boundaries: written by the general align kernel only, so
  // small batches pass no table and their GEMMs skip the lookup altogether
  long long* sched = (MK <= 32 || (h->step_cost[0] == 0 && h->step_cost[1] == 0))
                         ? nullptr
                         : reinterpret_cast<long long*>(ws + L.sched);
  aa.sched = sched;
  aa.sched_ctas = h->num_ctas;
  aa.sched_R[0] = 2 * h->N / kBM;
  aa.sched_KBn[0] = h->K / (2 * kBK);
  aa.sched_R[1] = h->K / kBM;
  aa.sched_KBn[1] = h->N / (2 * kBK);
  aa.step_cost_per_group[0] = h->step_cost[0];
  aa.step_cost_per_group[1] = h->step_cost[1];

  GatherArgs ga{};
  ga.x = hidden;
  ga.sorted_ids = sorted;
  ga.hdr = hdr;
  ga.MK = static_cast<int>(MK);
  ga.topk = h->topk;
  ga.K = h->K;
  ga.Gcap = L.Gcap;
  ga.xs = xs;
  ga.rowexp = rowexp;
  ga.acc = acc;
  ga.acc_elems = static_cast<long long>(M) * h->K;
  ga.xs_bytes = static_cast<long long>(L.Pcap) * h->K * 2;
  ga.M = M;
  ga.dbg = hdr + 8;
  ga.perm1 = h->perm1;
  ga.topk_ids = topk_ids;
  ga.e_begin = h->e_begin;
  // Small batch with given ids: both GEMMs in one cooperative launch that also
  // routes and gathers for itself (its gate/up shares start at multiples of 4
  // steps, so the steps per unit must allow that; at most one CTA per SM).
  const bool fused = h->fused_small && MK <= 32 && !logits && h->num_ctas <= h->num_sms &&
                     (static_cast<long long>(2 * h->N / kBM) * (h->K / (2 * kBK))) % 4 == 0;
  // Otherwise both products as CUDA-core matrix-vector products (tiles of at most
  // 4 token rows per expert): by default for batches of at most 256 routed slots
  // (measured faster there than the tensor-core kernels), else on the tensor cores.
  // (their split tables hold step indices as int: at most MK tiles x 2N/128 row tiles x K/128 steps)
  const bool gemv_wanted = h->gemv_small == 1 ? MK <= kGemvDefaultSlots
                           : h->gemv_small == 2 ? M == 1
                           : h->gemv_small == 3 ? MK <= kGemvMaxSlots : false;
  const bool gemv = !fused && gemv_wanted && MK * static_cast<long long>(2 * h->N / kBM) * (h->K / 128) < (1LL << 31);
  // ... and for at most 32 routed slots both of them in one cooperative launch (at
  // most one CTA per SM; the intermediate's step rows are handed over between CTAs
  // through counters in the ticket area, which the routing kernel zeroes)
  const bool gemv_one = gemv && MK <= 32 && h->gemv_one_launch && h->num_ctas <= h->num_sms;
  uint8_t* xv1 = ws + L.xv1;
  uint8_t* xv2 = ws + L.xv2;
  GemvTile* gv_tiles = reinterpret_cast<GemvTile*>(ws + L.gv_tiles);
  const long long xv1_bytes = MK * static_cast<long long>(h->K / 128) * kXvStepBytes;
  const long long xv2_bytes = MK * static_cast<long long>(h->N / 128) * kXvStepBytes;
  if (gemv) {
    ga.xv = xv1;
    ga.xv_steps = h->K / 128;
    ga.xs_bytes = xv1_bytes;  // (the extent the rows are written into)
    if (MK > 32) {            // the align kernel writes the tile list
      aa.gv_tiles = gv_tiles;
      aa.gv_tiles_cap = static_cast<int>(MK);
    }
  }
  if (fused) {
    if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[1], s));
  } else if (MK <= 32) {
    // small batch (decode): routing and gather in one launch, timed as "align"
    MOE_CUDA_TRY(launch_route_gather_small(aa, ga, L.Pcap, h->num_sms, s, false));
    if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[1], s));
  } else {
    if (logits)  // router kernel first; the align reads what it wrote
      MOE_CUDA_TRY(launch_route(logits, M, h->E_total, h->topk, const_cast<int32_t*>(topk_ids),
                                const_cast<float*>(topk_weights), h->num_sms, s, false));
    MOE_CUDA_TRY(launch_align(aa, s, logits != nullptr && pdl));
    if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[1], s));
    MOE_CUDA_TRY(launch_gather(ga, L.Gcap, h->num_sms, s, pdl));
  }
  if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[2], s));

  GemmArgs g1{};
  g1.wpack = h->w1p;
  g1.bsrc = xs;
  g1.hdr = hdr;
  g1.tiles = tiles;
  g1.expert_tiles = expert_tiles;
  g1.rowexp = rowexp;
  g1.wait_kcycles = wait_limit_kcycles(h->wait_us);
  g1.test_never_wait = h->test_never_wait ? 1 : 0;
  // a small batch whose ids are an input: the GEMMs recompute its routing tiles and
  // start their weight streams without waiting for the routing + gather launch
  const int32_t* small_ids = (MK <= 32 && !logits) ? topk_ids : nullptr;
  g1.small_ids = small_ids;
  if (gemv && MK > 32) {
    g1.small_ids = nullptr;
    g1.gv_tiles = gv_tiles;
  }
  if (gemv) {
    // a small batch: the CUDA-core kernels route from the ids themselves (routed
    // in-launch, they are the preceding kernel's output); a larger one reads the
    // align kernel's tile list
    if (MK <= 32) {
      g1.small_ids = topk_ids;
      g1.ids_after_pdl = logits ? 1 : 0;
    }
    g1.xv_in = xv1;
    g1.xv_bytes = xv1_bytes;
    g1.xv_out = xv2;
    g1.xv_out_bytes = xv2_bytes;
    g1.Pcap = L.Pcap;
  }
  g1.e_begin = h->e_begin;
  g1.E_total = h->E_total;
  g1.R = 2 * h->N / kBM;
  g1.KBn = h->K / (2 * kBK);  // GEMM pipeline steps of 128 reduction elements
  g1.Gcap = L.Gcap;
  g1.hout = hbuf;
  g1.scratch = scratch;
  g1.tickets = tickets;
  g1.MK = static_cast<int>(MK);
  g1.topk = h->topk;
  g1.status = hdr + kHdrStatus;
  g1.wpack_bytes = static_cast<long long>(h->w1p_bytes);
  g1.bsrc_bytes = static_cast<long long>(L.Pcap) * h->K * 2;
  g1.hout_bytes = static_cast<long long>(L.Pcap) * h->N * 2;
  g1.scratch_elems = static_cast<long long>(h->num_ctas) * 2 * kBNMax * kBM;
  g1.sorted_cap = L.Pcap;
  g1.tiles_cap = L.Gcap;
  g1.E = h->E;
  g1.dbg = hdr + 8;
  g1.sched = (sched && h->step_cost[0] > 0) ? sched : nullptr;
  if (gemv) {
    if (!gemv_one) MOE_CUDA_TRY(launch_gemv_gateup(g1, h->num_ctas, s, pdl));
  } else if (!fused)
    MOE_CUDA_TRY(launch_gemm_gateup(g1, h->num_ctas, s, pdl));
  if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[3], s));

  GemmArgs g2{};
  g2.wpack = h->w2p;
  g2.bsrc = hbuf;
  g2.hdr = hdr;
  g2.tiles = tiles;
  g2.expert_tiles = expert_tiles;
  g2.rowexp = rowexp;
  g2.wait_kcycles = wait_limit_kcycles(h->wait_us);
  g2.test_never_wait = h->test_never_wait ? 1 : 0;
  g2.small_ids = small_ids;
  g2.e_begin = h->e_begin;
  g2.E_total = h->E_total;
  g2.R = h->K / kBM;
  g2.KBn = h->N / (2 * kBK);
  g2.Gcap = L.Gcap;
  g2.sorted_ids = sorted;
  g2.topk_weights = topk_weights;
  g2.acc = acc;
  g2.Kout = h->K;
  g2.MK = static_cast<int>(MK);
  g2.topk = h->topk;
  g2.status = hdr + kHdrStatus;
  g2.wpack_bytes = static_cast<long long>(h->w2p_bytes);
  g2.bsrc_bytes = static_cast<long long>(L.Pcap) * h->N * 2;
  g2.acc_elems = static_cast<long long>(M) * h->K;
  g2.sorted_cap = L.Pcap;
  g2.tiles_cap = L.Gcap;
  g2.E = h->E;
  g2.dbg = hdr + 8;
  g2.sched = (sched && h->step_cost[1] > 0) ? sched + (h->num_ctas + 1) : nullptr;
  if (gemv) {
    g2.small_ids = MK <= 32 ? topk_ids : nullptr;
    g2.ids_after_pdl = (MK <= 32 && logits) ? 1 : 0;
    g2.gv_tiles = MK <= 32 ? nullptr : gv_tiles;
    g2.xv_in = xv2;
    g2.xv_bytes = xv2_bytes;
    g2.Pcap = L.Pcap;
  }
  if (fused) {
    // the counters live in the handle (zero between calls); the kernel writes the
    // workspace header itself at the end
    int32_t* fs = h->fsync;
    g1.status = g2.status = fs + kFsStatus;
    g1.tickets = fs + kFsTickets;
    g1.h_ready = g2.h_ready = fs + kFsTickets + kMaxCtas + h->K / kBM;
    FusedPrep& P = g1.prep;
    P.x = hidden;
    P.xs = xs;
    P.sorted_ids = sorted;
    P.rowexp = rowexp;
    P.acc = acc;
    P.acc_elems = static_cast<long long>(M) * h->K;
    P.perm1 = h->perm1;
    P.fsync = fs;
    P.fsync_words = h->fsync_words;
    P.ws_hdr = hdr;
    P.K = h->K;
    P.topk = h->topk;
    g2.prep = P;
    MOE_CUDA_TRY(launch_gemm_fused(g1, g2, h->num_ctas, s, false));
  } else if (gemv_one) {
    // the counters after the split-unit tickets and the row-tile words:
    // [kSmallTiles][N/128], one per tile and down step
    g1.h_ready = g2.h_ready = tickets + kMaxCtas + h->K / kBM;
    cudaError_t e = launch_gemv_both(g1, g2, h->num_ctas, s, pdl);
    if (e != cudaSuccess && pdl) {
      // (should the driver refuse a cooperative launch with programmatic
      // dependence: launch it after the routing kernel instead)
      (void)cudaGetLastError();
      e = launch_gemv_both(g1, g2, h->num_ctas, s, false);
    }
    MOE_CUDA_TRY(e);
  } else if (gemv) {
    MOE_CUDA_TRY(launch_gemv_down(g2, h->num_ctas, s, pdl));
  } else {
    MOE_CUDA_TRY(launch_gemm_down(g2, h->num_ctas, s, pdl));
  }
  if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[4], s));

  if (!partial)
    MOE_CUDA_TRY(launch_finalize(acc, out, static_cast<long long>(M) * h->K, h->num_sms, s, pdl));
  if (prof) MOE_CUDA_TRY(cudaEventRecord(h->ev[5], s));
  return MOE_W4A16_OK;
}

}  // namespace

extern "C" {

int moe_w4a16_forward(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                      const float* topk_weights, uint16_t* out, int M, void* workspace,
                      size_t workspace_bytes, void* stream) {
  return forward_impl(h, hidden, nullptr, topk_ids, topk_weights, out, M, workspace, workspace_bytes,
                      stream);
}

int moe_w4a16_forward_logits(moe_w4a16_t h, const uint16_t* hidden, const float* router_logits,
                             int32_t* topk_ids, float* topk_weights, uint16_t* out, int M,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!router_logits && M > 0) return fail(MOE_W4A16_INVALID_ARG, "null router_logits");
  return forward_impl(h, hidden, router_logits, topk_ids, topk_weights, out, M, workspace,
                      workspace_bytes, stream);
}

int moe_w4a16_forward_partial(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                              const float* topk_weights, float* partial, int M, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!partial && M > 0) return fail(MOE_W4A16_INVALID_ARG, "null partial");
  return forward_impl(h, hidden, nullptr, topk_ids, topk_weights, nullptr, M, workspace,
                      workspace_bytes, stream, partial);
}

int moe_w4a16_finalize(const float* acc, uint16_t* out, long long n, void* stream) {
  if (n < 0) return fail(MOE_W4A16_INVALID_ARG, "n must be >= 0");
  if (n == 0) return MOE_W4A16_OK;
  if (!acc || !out) return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  if ((reinterpret_cast<uintptr_t>(acc) | reinterpret_cast<uintptr_t>(out)) % 16 != 0 || n % 8 != 0)
    return fail(MOE_W4A16_INVALID_ARG, "acc and out must be 16-byte aligned and n a multiple of 8");
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  MOE_CUDA_TRY(launch_finalize(acc, out, n, sms, static_cast<cudaStream_t>(stream), false));
  return MOE_W4A16_OK;
}

int moe_w4a16_route(const float* router_logits, int M, int E, int topk, int32_t* topk_ids,
                    float* topk_weights, void* stream) {
  if (M < 0 || E < 1 || E > kMaxExperts || topk < 1 || topk > E)
    return fail(MOE_W4A16_INVALID_ARG, "bad shape (need M >= 0, 1 <= topk <= E <= 1024)");
  if (topk > 32) return fail(MOE_W4A16_UNSUPPORTED_SHAPE, "the router supports topk <= 32");
  if (M == 0) return MOE_W4A16_OK;
  if (!router_logits || !topk_ids || !topk_weights) return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  int dev = 0, sms = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  MOE_CUDA_TRY(launch_route(router_logits, M, E, topk, topk_ids, topk_weights, sms,
                            static_cast<cudaStream_t>(stream), false));
  return MOE_W4A16_OK;
}

int moe_w4a16_forward_host(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                           const float* topk_weights, uint16_t* out, int M, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (M < 0) return fail(MOE_W4A16_INVALID_ARG, "M must be >= 0");
  if (M == 0) return MOE_W4A16_OK;
  if (!hidden || !topk_ids || !topk_weights || !out || !workspace)
    return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  const size_t need = ws_layout(h, M).total;
  const size_t stage = staging_bytes(h, M);
  if (workspace_bytes < need + stage)
    return fail(MOE_W4A16_WORKSPACE_TOO_SMALL,
                "workspace too small: need " + std::to_string(need + stage) + " bytes");
  auto s = static_cast<cudaStream_t>(stream);
  // device staging after the workspace (batches moved by the copy engines):
  // [hidden | ids | weights | out]
  uint8_t* st = static_cast<uint8_t*>(workspace) + need;
  const size_t xb = static_cast<size_t>(M) * h->K * 2, rb = static_cast<size_t>(M) * h->topk * 4;
  const size_t xa = align_up(xb, 256), ra = align_up(rb, 256), in_bytes = xa + 2 * ra;
  uint16_t* d_x = reinterpret_cast<uint16_t*>(st);
  int32_t* d_ids = reinterpret_cast<int32_t*>(st + xa);
  float* d_w = reinterpret_cast<float*>(st + xa + ra);
  uint16_t* d_out = reinterpret_cast<uint16_t*>(st + in_bytes);

  // Small batches: zero-copy. The kernels read the inputs from, and the finalize
  // kernel writes the output to, pinned host memory: the caller's buffers when
  // they are pinned, else the handle's pinned staging block. This spares the copy
  // engines' per-transfer latency, which at decode sizes exceeds the transfer.
  if (xb <= kZeroCopyMaxBytes) {
    const void* px = pinned_device_pointer(hidden);
    const void* pi = px ? pinned_device_pointer(topk_ids) : nullptr;
    const void* pw = pi ? pinned_device_pointer(topk_weights) : nullptr;
    const void* po = pw ? pinned_device_pointer(out) : nullptr;
    if (po && ((reinterpret_cast<uintptr_t>(px) | reinterpret_cast<uintptr_t>(po)) % 16) == 0) {
      if (int rc = moe_w4a16_forward(h, static_cast<const uint16_t*>(px), static_cast<const int32_t*>(pi),
                                     static_cast<const float*>(pw), static_cast<uint16_t*>(const_cast<void*>(po)),
                                     M, workspace, need, stream))
        return rc;
      MOE_CUDA_TRY(cudaStreamSynchronize(s));
      return MOE_W4A16_OK;
    }
    // pageable buffers: [hidden | ids | weights | out] in the pinned staging block
    if (h->hstage_bytes < in_bytes + xa) {
      if (h->hstage) cudaFreeHost(h->hstage);
      h->hstage = nullptr;
      h->hstage_bytes = 0;
      MOE_CUDA_TRY(cudaHostAlloc(reinterpret_cast<void**>(&h->hstage), in_bytes + xa, cudaHostAllocMapped));
      h->hstage_bytes = in_bytes + xa;
    }
    uint8_t* hs = h->hstage;
    void* dev = nullptr;
    MOE_CUDA_TRY(cudaHostGetDevicePointer(&dev, hs, 0));
    uint8_t* ds = static_cast<uint8_t*>(dev);
    std::memcpy(hs, hidden, xb);
    std::memcpy(hs + xa, topk_ids, rb);
    std::memcpy(hs + xa + ra, topk_weights, rb);
    if (int rc = moe_w4a16_forward(h, reinterpret_cast<const uint16_t*>(ds), reinterpret_cast<const int32_t*>(ds + xa),
                                   reinterpret_cast<const float*>(ds + xa + ra),
                                   reinterpret_cast<uint16_t*>(ds + in_bytes), M, workspace, need, stream))
      return rc;
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    std::memcpy(out, hs + in_bytes, xb);
    return MOE_W4A16_OK;
  }

  MOE_CUDA_TRY(cudaMemcpyAsync(d_x, hidden, xb, cudaMemcpyHostToDevice, s));
  MOE_CUDA_TRY(cudaMemcpyAsync(d_ids, topk_ids, rb, cudaMemcpyHostToDevice, s));
  MOE_CUDA_TRY(cudaMemcpyAsync(d_w, topk_weights, rb, cudaMemcpyHostToDevice, s));
  if (int rc = moe_w4a16_forward(h, d_x, d_ids, d_w, d_out, M, workspace, need, stream)) return rc;
  MOE_CUDA_TRY(cudaMemcpyAsync(out, d_out, xb, cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  return MOE_W4A16_OK;
}

int moe_w4a16_status(moe_w4a16_t h, const void* workspace, int32_t* status, void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!workspace || !status) return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  auto s = static_cast<cudaStream_t>(stream);
  MOE_CUDA_TRY(cudaMemcpyAsync(status, static_cast<const uint8_t*>(workspace), sizeof(int32_t),
                               cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  return MOE_W4A16_OK;
}

int moe_w4a16_read_intermediate(moe_w4a16_t h, const void* workspace, int M, float* h_rows,
                                void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!workspace || !h_rows || M <= 0) return fail(MOE_W4A16_INVALID_ARG, "bad argument");
  const WsLayout L = ws_layout(h, M);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  MOE_CUDA_TRY(launch_read_intermediate(ws + L.hbuf, reinterpret_cast<const int32_t*>(ws + L.sorted),
                                        reinterpret_cast<const int32_t*>(ws + L.rowexp),
                                        reinterpret_cast<const int32_t*>(ws + L.hdr), M * h->topk,
                                        h->N, L.Gcap, L.Pcap, h_rows,
                                        static_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

int moe_w4a16_read_accumulator(moe_w4a16_t h, const void* workspace, int M, float* acc,
                               void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!workspace || !acc || M <= 0) return fail(MOE_W4A16_INVALID_ARG, "bad argument");
  const WsLayout L = ws_layout(h, M);
  MOE_CUDA_TRY(cudaMemcpyAsync(acc, static_cast<const uint8_t*>(workspace) + L.acc,
                               static_cast<size_t>(M) * h->K * sizeof(float), cudaMemcpyDeviceToDevice,
                               static_cast<cudaStream_t>(stream)));
  return MOE_W4A16_OK;
}

int moe_w4a16_schedule_debug(moe_w4a16_t h, const void* workspace, int M, int64_t* bounds, int n,
                             int* flags, void* stream) {
  if (int rc = check_handle(h)) return rc;
  if (!workspace || !bounds || !flags || M <= 0) return fail(MOE_W4A16_INVALID_ARG, "bad argument");
  if (n < 2 * (h->num_ctas + 1)) return fail(MOE_W4A16_INVALID_ARG, "bounds holds fewer than 2 * (ctas + 1) entries");
  const WsLayout L = ws_layout(h, M);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  auto s = static_cast<cudaStream_t>(stream);
  int32_t hdr[kHdrWords];
  MOE_CUDA_TRY(cudaMemcpyAsync(hdr, ws + L.hdr, sizeof(hdr), cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaMemcpyAsync(bounds, ws + L.sched, 2 * (h->num_ctas + 1) * sizeof(int64_t),
                               cudaMemcpyDeviceToHost, s));
  MOE_CUDA_TRY(cudaStreamSynchronize(s));
  *flags = hdr[kHdrSched];
  return 2 * (h->num_ctas + 1);
}

int moe_w4a16_align_debug(const int32_t* topk_ids, int M, int topk, int E, int block,
                          int32_t* sorted_ids, int32_t* expert_offsets, int32_t* num_padded,
                          int capacity, void* stream) {
  if (M < 0 || topk < 1 || E < 1 || E > kMaxExperts || block < 1)
    return fail(MOE_W4A16_INVALID_ARG, "bad shape");
  if ((M > 0 && !topk_ids) || !sorted_ids || !expert_offsets || !num_padded)
    return fail(MOE_W4A16_INVALID_ARG, "null pointer argument");
  const long long MK = static_cast<long long>(M) * topk;
  const long long active = MK < E ? MK : E;
  if (capacity < MK + active * (block - 1))
    return fail(MOE_W4A16_INVALID_ARG, "capacity too small");
  AlignArgs aa{};
  aa.topk_ids = topk_ids;
  aa.MK = static_cast<int>(MK);
  aa.E = E;
  aa.E_total = E;
  aa.block = block;
  aa.bn_max = 0;
  aa.sorted_ids = sorted_ids;
  aa.expert_offsets = expert_offsets;
  aa.num_padded_out = num_padded;
  MOE_CUDA_TRY(align_set_attributes(E));
  MOE_CUDA_TRY(launch_align(aa, static_cast<cudaStream_t>(stream), false));
  return MOE_W4A16_OK;
}

}  // extern "C"
