// Token->expert align, expert-sorted gather of the hidden states, output
// finalisation and the intermediate-activation readback used by tests.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kernels.cuh"
#include "rowcopy.cuh"
#include "route.cuh"
#include "small_route.cuh"

namespace moe {

// Exclusive prefix sum over the 1024 threads of the block; *total gets the sum.
__device__ int block_exclusive_scan(int v, int* warp_tmp, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tmp[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nwarps ? warp_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tmp[lane] = t;  // inclusive per-warp totals
  }
  __syncthreads();
  const int before = (w > 0 ? warp_tmp[w - 1] : 0) + x - v;
  *total = warp_tmp[nwarps - 1];
  __syncthreads();
  return before;
}

// One CTA of 1024 threads. Every warp owns a contiguous chunk of the flat slot
// list, histograms it privately, and then scatters its chunk in order, so the
// result is the stable counting sort: for each expert in id order, the flat slot
// ids routed to it in ascending order, padded with the sentinel MK to a
// multiple of `block`.
__global__ void __launch_bounds__(1024) align_kernel(const AlignArgs a) {
  extern __shared__ int sm[];
  const int E = a.E;
  int* hist = sm;  // [32][E]: per-warp counts, then per-warp start offsets
  __shared__ int warp_tmp[32];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0 && a.hdr) {
    a.hdr[kHdrStatus] = 0;
    a.hdr[kHdrSched] = 0;
  }
  if (tid < 8 && a.dbg) a.dbg[tid] = 0;
  for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
  if (a.tickets)
    for (int i = tid; i < a.n_tickets; i += blockDim.x) a.tickets[i] = 0;
  __syncthreads();

  const int chunk = (a.MK + 31) / 32;
  const int lo = min(a.MK, w * chunk), hi = min(a.MK, lo + chunk);
  int bad = 0;
  for (int i = lo + lane; i < hi; i += 32) {
    bool b = false;
    const int e = local_expert(a.topk_ids[i], a.e_begin, E, a.E_total, &b);
    if (e >= 0) atomicAdd(&hist[w * E + e], 1);
    bad |= b ? 1 : 0;
  }
  if (bad && a.hdr) atomicOr(&a.hdr[kHdrStatus], 1);
  __syncthreads();

  int my_cnt = 0, my_pad = 0, my_tiles = 0;
  if (tid < E) {
    int run = 0;
    for (int ww = 0; ww < 32; ++ww) {
      const int c = hist[ww * E + tid];
      hist[ww * E + tid] = run;
      run += c;
    }
    my_cnt = run;
    my_pad = (run + a.block - 1) / a.block * a.block;
    my_tiles = a.bn_max > 0 ? (my_pad + a.bn_max - 1) / a.bn_max : 0;
  }
  int tot_pad = 0, tot_tiles = 0, tot_gv = 0;
  const int seg = block_exclusive_scan(my_pad, warp_tmp, &tot_pad);
  const int tstart = block_exclusive_scan(my_tiles, warp_tmp, &tot_tiles);
  const int my_gv = (my_cnt + kGemvRows - 1) / kGemvRows;  // (0 for threads beyond E)
  const int gstart = a.gv_tiles ? block_exclusive_scan(my_gv, warp_tmp, &tot_gv) : 0;
  int* seg_sm = hist + 32 * E;  // [E]
  if (tid < E) seg_sm[tid] = seg;
  __syncthreads();

  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    int e = -1;
    if (i < hi) {
      bool b = false;
      e = local_expert(a.topk_ids[i], a.e_begin, E, a.E_total, &b);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = seg_sm[e] + hist[w * E + e] + rank;
      if (MOE_CHECK(a.sorted_cap <= 0 || pos < a.sorted_cap, a.hdr, a.dbg, 21, pos, e))
        a.sorted_ids[pos] = i;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) hist[w * E + e] += __popc(peers);
    __syncwarp();
  }

  if (tid < E) {
    for (int p = seg + my_cnt; p < seg + my_pad; ++p)
      if (MOE_CHECK(a.sorted_cap <= 0 || p < a.sorted_cap, a.hdr, a.dbg, 22, p, tid))
        a.sorted_ids[p] = a.MK;
    if (a.expert_offsets) {
      a.expert_offsets[tid] = seg;
      if (tid == E - 1) a.expert_offsets[E] = tot_pad;
    }
    if (a.bn_max > 0) {
      for (int t = 0; t < my_tiles; ++t) {
        TokenTile tt;
        tt.expert = tid;
        tt.g0 = (seg + t * a.bn_max) / kRowGroup;
        tt.ngroups = min(a.bn_max, my_pad - t * a.bn_max) / kRowGroup;
        tt.first = tstart;
        if (MOE_CHECK(tstart + t < a.tiles_cap, a.hdr, a.dbg, 23, tstart + t, tid))
          a.tiles[tstart + t] = tt;
      }
      a.expert_tiles[tid] = my_tiles;
    }
  }
  if (a.gv_tiles) {
    // the CUDA-core tiles: each expert's rows (now in sorted_ids) four at a time
    __syncthreads();
    if (tid < E) {
      for (int j = 0; j < my_gv; ++j) {
        GemvTile gt;
        gt.e = tid;
        gt.p0 = seg + j * kGemvRows;
        gt.n = min(kGemvRows, my_cnt - j * kGemvRows);
        gt.pad = 0;
#pragma unroll
        for (int t = 0; t < kGemvRows; ++t) gt.slot[t] = t < gt.n ? a.sorted_ids[gt.p0 + t] : a.MK;
        if (MOE_CHECK(gstart + j < a.gv_tiles_cap, a.hdr, a.dbg, 30, gstart + j, tid)) a.gv_tiles[gstart + j] = gt;
      }
    }
  }
  if (tid == 0) {
    if (a.hdr) {
      a.hdr[kHdrNumPadded] = tot_pad;
      a.hdr[kHdrNumTiles] = tot_tiles;
      a.hdr[kHdrNumGemvTiles] = tot_gv;
    }
    if (a.num_padded_out) *a.num_padded_out = tot_pad;
  }

  // Cost-weighted stream-K boundaries, per GEMM. Each GEMM's steps run in unit
  // order [expert][row tile][token tile of the expert]; a step of a unit whose
  // token tile has ng row groups costs step_cost(ng, c) with that GEMM's c. CTA j
  // starts at the first step where the cost so far reaches j/G of the total, so
  // CTAs that draw a hot expert's full 64-row tiles get fewer steps. A GEMM with
  // c = 0 keeps the even split (its header bit stays clear).
  if (a.sched != nullptr && a.bn_max > 0) {
    long long* Pe = reinterpret_cast<long long*>(hist);  // [E + 1] cost before expert e's tiles
    int* fe = reinterpret_cast<int*>(Pe + E + 1);        // [E] first tile
    int* tee = fe + E;                                   // [E] tiles
    int* cle = tee + E;                                  // [E] step cost of the last tile
    const int G = a.sched_ctas;
    int bits = 0;
    for (int w = 0; w < 2; ++w) {
      const int cpg = a.step_cost_per_group[w];
      if (cpg <= 0) continue;  // uniform across the block
      bits |= 1 << w;
      __syncthreads();  // the histograms, or the previous GEMM's costs, are no longer read
      const int cfull = step_cost(a.bn_max / kRowGroup, cpg);
      int my_cost = 0, c_last = 0;
      if (tid < E && my_tiles > 0) {
        c_last = step_cost((my_pad - (my_tiles - 1) * a.bn_max) / kRowGroup, cpg);
        my_cost = (my_tiles - 1) * cfull + c_last;
      }
      int tot_cost = 0;
      const int before = block_exclusive_scan(my_cost, warp_tmp, &tot_cost);
      if (tid < E) {
        Pe[tid] = before;
        fe[tid] = tstart;
        tee[tid] = my_tiles;
        cle[tid] = c_last;
      }
      if (tid == 0) Pe[E] = tot_cost;
      __syncthreads();
      const long long R = a.sched_R[w], KB = a.sched_KBn[w];
      const long long W = static_cast<long long>(tot_tiles) * R * KB;
      for (int c = tid; c <= G; c += blockDim.x) {
        long long g = 0;
        if (c == G) {
          g = W;
        } else if (tot_cost > 0) {
          const long long T = static_cast<long long>(c) * tot_cost * R * KB / G;
          int lo = 0, hi = E - 1;  // the last expert whose tiles start at cost <= T
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (KB * R * Pe[mid] <= T)
              lo = mid;
            else
              hi = mid - 1;
          }
          const int e = lo;
          const long long T1 = T - KB * R * Pe[e];
          const long long Ce = Pe[e + 1] - Pe[e];  // > 0: T lies inside expert e's units
          const long long rt = T1 / (KB * Ce);
          const long long T2 = T1 - rt * KB * Ce;
          const int te = tee[e];
          long long tt = T2 / (KB * cfull);  // every tile but the last is full
          if (tt > te - 1) tt = te - 1;
          const long long T3 = T2 - tt * KB * cfull;
          const long long ct = (tt == te - 1) ? cle[e] : cfull;
          long long kb = (T3 + ct - 1) / ct;
          if (kb > KB) kb = KB;
          g = (R * fe[e] + rt * te + tt) * KB + kb;
          if (g > W) g = W;
        }
        a.sched[w * (G + 1) + c] = g;
      }
    }
    if (tid == 0 && a.hdr) a.hdr[kHdrSched] = bits;
  }
  pdl_launch_dependents();
}

__device__ SmallRoute small_route(const AlignArgs& a, int lane) {
  return small_route(a.topk_ids, a.MK, a.E, a.block, a.bn_max, lane, a.e_begin, a.E_total);
}

// Write the routing outputs of a small batch (one warp): header, counters, sorted
// slot ids, token tiles, and (debug entry) the offsets of all E experts.
__device__ void small_route_write(const AlignArgs& a, const SmallRoute& r, int lane) {
  // header first: the range checks below may OR bits into the status word
  if (lane == 0) {
    if (a.hdr) {
      a.hdr[kHdrStatus] = r.any_bad ? 1 : 0;
      a.hdr[kHdrNumPadded] = r.tot_pad;
      a.hdr[kHdrNumTiles] = r.tot_tiles;
      a.hdr[kHdrSched] = 0;  // at most 32 routed rows: an even split of the steps
    }
    if (a.num_padded_out) *a.num_padded_out = r.tot_pad;
  }
  if (lane < 8 && a.dbg) a.dbg[lane] = 0;
  if (a.tickets)
    for (int i = lane; i < a.n_tickets; i += 32) a.tickets[i] = 0;
  __syncwarp();
  if (r.e >= 0 &&
      MOE_CHECK(a.sorted_cap <= 0 || r.seg + r.rank < a.sorted_cap, a.hdr, a.dbg, 26, r.seg + r.rank, r.e))
    a.sorted_ids[r.seg + r.rank] = lane;
  if (r.leader) {
    for (int p = r.seg + r.cnt; p < r.seg + r.pad; ++p)
      if (MOE_CHECK(a.sorted_cap <= 0 || p < a.sorted_cap, a.hdr, a.dbg, 27, p, r.e))
        a.sorted_ids[p] = a.MK;
    if (a.bn_max > 0) {
      for (int t = 0; t < r.ntile; ++t) {
        TokenTile tt;
        tt.expert = r.e;
        tt.g0 = (r.seg + t * a.bn_max) / kRowGroup;
        tt.ngroups = min(a.bn_max, r.pad - t * a.bn_max) / kRowGroup;
        tt.first = r.tile0;
        if (MOE_CHECK(r.tile0 + t < a.tiles_cap, a.hdr, a.dbg, 28, r.tile0 + t, r.e))
          a.tiles[r.tile0 + t] = tt;
      }
      a.expert_tiles[r.e] = r.ntile;
    }
  }
  if (a.expert_offsets) {
    const int lead_e = r.leader ? r.e : -1;
    for (int x0 = 0; x0 <= a.E; x0 += 32) {  // uniform trip count: shuffles stay converged
      const int x = x0 + lane;
      int off = 0;
      for (int j = 0; j < 32; ++j) {
        const int ej = __shfl_sync(0xffffffffu, lead_e, j);
        const int pj = __shfl_sync(0xffffffffu, r.pad, j);
        if (ej >= 0 && ej < x) off += pj;
      }
      if (x <= a.E) a.expert_offsets[x] = off;
    }
  }
}

__global__ void __launch_bounds__(32) align_small_kernel(const AlignArgs a) {
  pdl_wait();
  const SmallRoute r = small_route(a, threadIdx.x);
  small_route_write(a, r, threadIdx.x);
  pdl_launch_dependents();
}

cudaError_t align_set_attributes(int E) {
  (void)E;
  // the limit covers every expert count a handle may have, so it is set once and
  // never again inside a forward (which may be under stream capture)
  return cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(33 * kMaxExperts * sizeof(int)));
}

cudaError_t launch_align(const AlignArgs& a, cudaStream_t stream, bool pdl) {
  if (a.MK <= 32) return launch_k(align_small_kernel, dim3(1), dim3(32), 0, stream, pdl, a);
  const size_t smem = (33 * static_cast<size_t>(a.E)) * sizeof(int);
  return launch_k(align_kernel, dim3(1), dim3(1024), smem, stream, pdl, a);
}

// One CTA copies expert-sorted row p (flat slot `sid`, or padding when sid is the
// sentinel) into the blocked fp16 B-operand layout: every thread loads its
// 16-byte chunks of the token's row at once (up to kGatherChunks each), the CTA
// reduces the row's largest magnitude, records the row's prescale exponent e and
// writes x * 2^-e. A padding row only gets the exponent kPadRowExp: its operand
// rows are never written (they only feed output columns that nothing reads, and
// the gate/up epilogue stores zeros for them).
constexpr int kGatherThreads = 256;
constexpr int kGatherChunks = 8;  // chunks of 8 elements per thread and pass: K <= 16384 in one pass
// With act-order on w1 (perm1 set) the row is written in the expert's packing
// order: element j of the copy is hidden element perm1[expert][j] (the largest
// magnitude, and so the exponent, does not depend on the order).
__device__ void gather_row(const GatherArgs& g, int p, int sid, int* red, int expert) {
  const int tid = threadIdx.x;
  const bool real = sid < g.MK && MOE_CHECK(sid >= 0 && sid / g.topk < g.M, const_cast<int32_t*>(g.hdr),
                                            g.dbg, 24, sid, p);
  if (!real) {  // uniform across the CTA
    if (tid == 0) g.rowexp[p] = kPadRowExp;
    return;
  }
  const int cpr = g.K / 8;  // 16-byte chunks per row
  const uint4* src = reinterpret_cast<const uint4*>(g.x + static_cast<long long>(sid / g.topk) * g.K);
  constexpr int kPass = kGatherThreads * kGatherChunks;
  const bool one_pass = cpr <= kPass;  // the whole row stays in registers (K <= 16384)
  uint4 v[kGatherChunks];
  uint32_t m = 0;
  for (int c0 = 0; c0 < cpr; c0 += kPass) {
#pragma unroll
    for (int i = 0; i < kGatherChunks; ++i) {
      const int ch = c0 + i * kGatherThreads + tid;
      v[i] = ch < cpr ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
      m = max(m, bf16x8_absmax_bits(v[i]));
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((tid & 31) == 0) red[tid >> 5] = static_cast<int>(m);
  __syncthreads();
  if (tid < 32) {
    uint32_t x = tid < kGatherThreads / 32 ? static_cast<uint32_t>(red[tid]) : 0u;
    x = __reduce_max_sync(0xffffffffu, x);
    if (tid == 0) red[kGatherThreads / 32] = static_cast<int>(x);
  }
  __syncthreads();
  const int e = row_exponent(static_cast<uint32_t>(red[kGatherThreads / 32]));
  __syncthreads();  // red is reused by the next row
  if (tid == 0) g.rowexp[p] = e;
  const float f = exp2_int(-e);
  const uint16_t* xr = g.x + static_cast<long long>(sid / g.topk) * g.K;
  const int32_t* pr = nullptr;
  if (g.perm1 && MOE_CHECK(expert >= 0, const_cast<int32_t*>(g.hdr), g.dbg, 26, expert, p))
    pr = g.perm1 + static_cast<long long>(expert) * g.K;
  for (int c0 = 0; c0 < cpr; c0 += kPass) {
#pragma unroll
    for (int i = 0; i < kGatherChunks; ++i) {
      const int ch = c0 + i * kGatherThreads + tid;
      const bool in_row = ch < cpr;  // (K is a multiple of 128: whole groups of 4 lanes agree)
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (in_row) {
        x = one_pass ? v[i] : src[ch];
        if (pr) {
          const int4 i0 = *reinterpret_cast<const int4*>(pr + 8 * ch);
          const int4 i1 = *reinterpret_cast<const int4*>(pr + 8 * ch + 4);
          x = make_uint4(bf16_pair(xr, i0.x, i0.y), bf16_pair(xr, i0.z, i0.w), bf16_pair(xr, i1.x, i1.y),
                         bf16_pair(xr, i1.z, i1.w));
        }
      }
      if (g.xv) {
        // step rows (layout.cuh): the chunk is one word of its scale group, whose
        // 4 words sit in 4 consecutive lanes; 16-bit block fixed point per group
        float xf[8];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xf[2 * k] = fminf(fmaxf(__uint_as_float(w[k] << 16) * f, -65504.0f), 65504.0f);
          xf[2 * k + 1] = fminf(fmaxf(__uint_as_float(w[k] & 0xFFFF0000u) * f, -65504.0f), 65504.0f);
          m = fmaxf(m, fmaxf(fabsf(xf[2 * k]), fabsf(xf[2 * k + 1])));
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int eg = xv_group_exp(m);
        uint16_t q[8];
        int sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int v16 = xv_quantize(xf[k], eg);
          q[xv_slot(k)] = static_cast<uint16_t>(v16);
          sum += v16;
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        uint8_t* xv_step = g.xv + (static_cast<long long>(sid) * g.xv_steps + (ch >> 4)) * kXvStepBytes;
        if (in_row && MOE_CHECK((xv_step - g.xv) + kXvStepBytes <= g.xs_bytes, const_cast<int32_t*>(g.hdr), g.dbg,
                                28, xv_step - g.xv, p)) {
          *reinterpret_cast<uint4*>(xv_step + (ch & 15) * 16) =
              make_uint4(q[0] | (static_cast<uint32_t>(q[1]) << 16), q[2] | (static_cast<uint32_t>(q[3]) << 16),
                         q[4] | (static_cast<uint32_t>(q[5]) << 16), q[6] | (static_cast<uint32_t>(q[7]) << 16));
          if ((ch & 3) == 0) xv_header(xv_step, (ch >> 2) & 3, sum, eg);
        }
      } else if (in_row) {
        const uint4 o = make_uint4(bf16x2_to_f16x2_scaled(x.x, f), bf16x2_to_f16x2_scaled(x.y, f),
                                   bf16x2_to_f16x2_scaled(x.z, f), bf16x2_to_f16x2_scaled(x.w, f));
        const long long off = b_operand_offset(ch, p, g.Gcap);
        if (MOE_CHECK(off + 16 <= g.xs_bytes, const_cast<int32_t*>(g.hdr), g.dbg, 25, off, p))
          *reinterpret_cast<uint4*>(g.xs + off) = o;
      }
    }
  }
}

// Small batches in one launch: routing and gather. Every CTA's first warp
// recomputes the one-warp routing (cheap) and lays the padded sorted-slot list
// into shared memory; CTA 0 also publishes the routing for the GEMMs (they read
// it after waiting for this kernel). Then CTA c >= 1 copies the row of routed slot
// c - 1 (the grid is only as large as the slots, or the accumulator to zero, need:
// every other SM is free for the GEMM launched behind it; CTA 0, which publishes,
// copies none), the padding rows get their sentinel exponent, and every thread
// zeroes its share of the accumulator.
#ifdef MOE_GEMM_TRACE
// trace builds: global-timer stamps per CTA (entry, dependency resolved, exit)
__device__ unsigned long long g_rg_trace[512][4];
extern "C" int moe_rg_trace_read(unsigned long long* host, int reset) {
  int e = static_cast<int>(cudaMemcpyFromSymbol(host, g_rg_trace, sizeof(g_rg_trace)));
  if (reset) {
    static unsigned long long z[512 * 4];
    cudaMemcpyToSymbol(g_rg_trace, z, sizeof(z));
  }
  return e;
}
#define RG_STAMP(ev)                                                                  \
  do {                                                                                \
    if (threadIdx.x == 0 && blockIdx.x < 512) {                                       \
      unsigned long long t;                                                           \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));                           \
      g_rg_trace[blockIdx.x][(ev)] = t;                                               \
    }                                                                                 \
  } while (0)
#else
#define RG_STAMP(ev) \
  do {               \
  } while (0)
#endif
constexpr int kGatherWarps = kGatherThreads / 32;

__global__ void __launch_bounds__(kGatherThreads) route_gather_small_kernel(const AlignArgs a_in,
                                                                           const GatherArgs g) {
  __shared__ int s_sorted[kSmallPadRows];
  __shared__ int s_expert[kSmallPadRows];  // expert of every real padded row
  __shared__ int s_pos[32];                // padded row of every routed slot, or -1
  __shared__ int s_npad;
  __shared__ int32_t s_ids[32];
  __shared__ int s_red[kGatherWarps + 1];
  RG_STAMP(0);
  pdl_wait();
  RG_STAMP(1);
  // The GEMM that follows starts its weight stream on its own; where it reads
  // this kernel's outputs it waits for this grid to complete. Let it launch now.
  pdl_launch_dependents();
  const AlignArgs& a = a_in;
  if (a.logits) {
    // route the (at most 32 / k) tokens first: warp w takes tokens w, w + 8, ...;
    // CTA 0 publishes ids and weights, every CTA keeps the ids in shared memory
    // for its own use (the published copy is written concurrently by CTA 0)
    const int lane = threadIdx.x & 31;
    for (int t = threadIdx.x >> 5; t < a.M_tokens; t += kGatherWarps) {
      int id;
      float w;
      warp_topk(a.logits + static_cast<long long>(t) * a.E_total, a.E_total, a.topk, lane, &id, &w);
      if (lane < a.topk) {
        s_ids[t * a.topk + lane] = id;
        if (blockIdx.x == 0) {
          a.ids_out[t * a.topk + lane] = id;
          a.wts_out[t * a.topk + lane] = w;
        }
      }
    }
    __syncthreads();
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int v = -1;  // this lane's slot id: from shared memory when routed here, else the input
    if (lane < a.MK) v = a.logits ? s_ids[lane] : a.topk_ids[lane];
    const SmallRoute r = small_route_ids(v, a.MK, a.E, a.block, a.bn_max, lane, a.e_begin, a.E_total);
    const int npad = r.tot_pad < kSmallPadRows ? r.tot_pad : kSmallPadRows;
    for (int p = lane; p < npad; p += 32) s_sorted[p] = a.MK;
    __syncwarp();
    const bool placed = r.e >= 0 && r.seg + r.rank < kSmallPadRows;
    if (placed) {
      s_sorted[r.seg + r.rank] = lane;
      s_expert[r.seg + r.rank] = r.e;
    }
    s_pos[lane] = placed ? r.seg + r.rank : -1;
    if (lane == 0) s_npad = npad;
    if (blockIdx.x == 0) small_route_write(a, r, lane);
  }
  __syncthreads();
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  float4* acc4 = reinterpret_cast<float4*>(g.acc);
  for (long long i = gt; i < g.acc_elems / 4; i += nthr) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // one CTA per routed slot copies its row (a small grid: the GEMM that follows
  // starts on every other SM at once), leaving CTA 0, which publishes the routing,
  // none when there are others; the padding rows only get their sentinel
  const int g0 = gridDim.x > 1 ? 1 : 0;
  for (int sl = static_cast<int>(blockIdx.x) - g0; sl >= 0 && sl < a.MK; sl += gridDim.x - g0) {
    const int p = s_pos[sl];
    if (p >= 0) gather_row(g, p, sl, s_red, s_expert[p]);
  }
  for (long long p = gt; p < s_npad; p += nthr)
    if (s_sorted[p] >= a.MK) g.rowexp[p] = kPadRowExp;
#ifdef MOE_GEMM_TRACE
  __syncthreads();
  RG_STAMP(2);
#endif
}

cudaError_t launch_route_gather_small(const AlignArgs& a, const GatherArgs& g, int max_rows,
                                      int num_sms, cudaStream_t stream, bool pdl) {
  (void)max_rows;
  const long long ctas = std::max<long long>(a.MK + 1, (g.acc_elems / 4 + kGatherThreads - 1) / kGatherThreads);
  long long grid = ctas;
  const long long cap = 4LL * num_sms;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_k(route_gather_small_kernel, dim3(static_cast<unsigned>(grid)), dim3(kGatherThreads), 0,
                  stream, pdl, a, g);
}

// Copy every expert-sorted row's hidden state, prescaled and as fp16, into the
// blocked B-operand layout, one CTA per row, and zero the fp32 output accumulator.
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const GatherArgs a) {
  __shared__ int s_red[kGatherWarps + 1];
  pdl_wait();
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  float4* acc4 = reinterpret_cast<float4*>(a.acc);
  for (long long i = gt; i < a.acc_elems / 4; i += nthr) acc4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int num_padded = a.hdr[kHdrNumPadded];
  for (int p = blockIdx.x; p < num_padded; p += gridDim.x) {
    const int sid = a.sorted_ids[p];
    // (the expert of a real row: align placed it in that expert's segment)
    const int e = a.perm1 && sid >= 0 && sid < a.MK ? a.topk_ids[sid] - a.e_begin : -1;
    gather_row(a, p, sid, s_red, e);
  }
  pdl_launch_dependents();
}

cudaError_t launch_gather(const GatherArgs& a, int max_groups, int num_sms, cudaStream_t stream,
                          bool pdl) {
  const long long rows = static_cast<long long>(max_groups) * kRowGroup;
  const long long ctas = std::max<long long>(rows, (a.acc_elems / 4 + kGatherThreads - 1) / kGatherThreads);
  long long grid = ctas;
  const long long cap = 8LL * num_sms;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_k(gather_kernel, dim3(static_cast<unsigned>(grid)), dim3(kGatherThreads), 0, stream,
                  pdl, a);
}

// out = bf16(acc), round to nearest even; eight elements per thread step.
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ acc,
                                                       uint16_t* __restrict__ out, long long n) {
  pdl_wait();
  const long long nthr = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  uint4* o4 = reinterpret_cast<uint4*>(out);
  for (long long i = gt; i < n / 8; i += nthr) {
    const float4 x = a4[2 * i], y = a4[2 * i + 1];
    __nv_bfloat162 p0 = __floats2bfloat162_rn(x.x, x.y);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(x.z, x.w);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(y.x, y.y);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(y.z, y.w);
    uint4 o;
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    o4[i] = o;
  }
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, long long n, int num_sms,
                            cudaStream_t stream, bool pdl) {
  long long blocks = (n / 8 + 255) / 256;
  const long long cap = 8LL * num_sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_k(finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, pdl,
                  acc, out, n);
}

__global__ void read_intermediate_kernel(const uint8_t* __restrict__ hbuf,
                                         const int32_t* __restrict__ sorted_ids,
                                         const int32_t* __restrict__ rowexp,
                                         const int32_t* __restrict__ hdr, int MK, int N, int Gcap,
                                         float* __restrict__ h_rows) {
  const int num_padded = hdr[kHdrNumPadded];
  for (int p = blockIdx.x; p < num_padded; p += gridDim.x) {
    const int sid = sorted_ids[p];
    if (sid >= MK) continue;
    int e = rowexp[p];  // (a real row: never the padding sentinel)
    e = e < -kMaxRowExp ? -kMaxRowExp : (e > kMaxRowExp ? kMaxRowExp : e);
    const float scale = exp2_int(2 * e);  // h was stored as h * 2^-2e
    const int g = p / kRowGroup, r = p % kRowGroup;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      const int kb = n >> 6, k = n & 63;
      const uint16_t bits = *reinterpret_cast<const uint16_t*>(
          hbuf + (static_cast<long long>(kb) * Gcap + g) * kRowGroupBytes + blocked_offset(r, k));
      h_rows[static_cast<long long>(sid) * N + n] = __half2float(__ushort_as_half(bits)) * scale;
    }
  }
}

cudaError_t launch_read_intermediate(const uint8_t* hbuf, const int32_t* sorted_ids,
                                     const int32_t* rowexp, const int32_t* hdr, int MK, int N,
                                     int Gcap, int max_rows, float* h_rows, cudaStream_t stream) {
  int grid = max_rows < 1024 ? (max_rows > 0 ? max_rows : 1) : 1024;
  read_intermediate_kernel<<<grid, 256, 0, stream>>>(hbuf, sorted_ids, rowexp, hdr, MK, N, Gcap,
                                                     h_rows);
  return cudaGetLastError();
}

}  // namespace moe
