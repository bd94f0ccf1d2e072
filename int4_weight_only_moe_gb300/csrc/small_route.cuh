// One-warp token->expert routing of a small batch (at most 32 routed slots),
// shared by the routing + gather kernel and by the GEMMs, which recompute it for
// themselves so that they can start streaming weights before the preceding kernel
// has finished.
#pragma once
#include <cstdint>

#include "layout.cuh"

namespace moe {

// Small batches (at most 32 routed slots, e.g. decode) take one warp, with no
// E-wide histograms, scans or block barriers: lane l holds flat slot l; lanes
// routed to the same expert find each other with __match_any_sync; a slot's rank
// among them counts the lower lanes (slot ids ascending, the same stable order as
// the general kernel); the padded segment and first tile of an expert add up the
// experts present (at most 32) with a smaller id. Experts without rows get no
// segment and no tiles (the GEMMs read only the tiles' experts).
struct SmallRoute {
  int e;          // this lane's expert, or -1 (no slot or a bad id)
  int rank, cnt;  // position among the slots of its expert, and their number
  bool leader;    // lowest lane of its expert
  int pad, ntile; // leader only: padded rows and token tiles of the expert
  int seg, tile0; // first padded row and first tile of the expert
  int tot_pad, tot_tiles;
  bool any_bad;
};

// `v` is the expert id of flat slot `lane` (read by the caller: global or shared
// memory), ignored for lanes at or beyond MK. The handle holds experts
// [e_begin, e_begin + E) of a layer of E_total: a slot of another expert of the
// layer is skipped, an id outside [0, E_total) is skipped and flagged.
__device__ __forceinline__ SmallRoute small_route_ids(int v, int MK, int E, int block, int bn_max,
                                                      int lane, int e_begin, int E_total) {
  SmallRoute r;
  r.e = -1;
  bool bad = false;
  if (lane < MK) r.e = local_expert(v, e_begin, E, E_total, &bad);
  const unsigned peers = __match_any_sync(0xffffffffu, r.e);
  const bool valid = r.e >= 0;
  r.rank = __popc(peers & ((1u << lane) - 1u));
  r.cnt = __popc(peers);
  r.leader = valid && r.rank == 0;
  r.pad = r.leader ? (r.cnt + block - 1) / block * block : 0;
  r.ntile = (r.leader && bn_max > 0) ? (r.pad + bn_max - 1) / bn_max : 0;
  const int lead_e = r.leader ? r.e : -1;
  r.seg = r.tile0 = r.tot_pad = r.tot_tiles = 0;
  for (int j = 0; j < 32; ++j) {
    const int ej = __shfl_sync(0xffffffffu, lead_e, j);
    const int pj = __shfl_sync(0xffffffffu, r.pad, j);
    const int tj = __shfl_sync(0xffffffffu, r.ntile, j);
    if (ej >= 0) {
      r.tot_pad += pj;
      r.tot_tiles += tj;
      if (ej < r.e) {
        r.seg += pj;
        r.tile0 += tj;
      }
    }
  }
  r.any_bad = __any_sync(0xffffffffu, bad);
  return r;
}

// The same, reading slot `lane`'s id from `ids` (global memory).
__device__ __forceinline__ SmallRoute small_route(const int32_t* ids, int MK, int E, int block,
                                                  int bn_max, int lane, int e_begin, int E_total) {
  return small_route_ids(lane < MK ? ids[lane] : -1, MK, E, block, bn_max, lane, e_begin, E_total);
}

}  // namespace moe
