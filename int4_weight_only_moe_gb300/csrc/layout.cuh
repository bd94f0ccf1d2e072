// Data layouts in device memory shared by the kernels and the host launcher.
//
// Packed weights (written once by the repack kernel). A GEMM operand W of shape
// [rows, Kred] (rows = output features) is cut into tiles of 128 rows and
// k-blocks of 64 reduction elements. Each (expert, row tile, k-block) is one
// contiguous 4608-byte block, so one bulk copy moves it into shared memory:
//
//   bytes [0, 4096):    codes, [half h (0..1)][row r (0..127)][4 words]; word j of
//                       (h, r) holds reduction elements 32h + 8j .. 32h + 8j + 7
//   bytes [4096, 4608): fp16 scales, [row r][half h]; half h is the scale group
//                       (both scales of a row in one 32-bit word)
//
// Inside a word the eight 4-bit codes are interleaved so that one shift and one
// mask put elements (2p, 2p+1) into the two 16-bit halves of a 32-bit register:
// element 2p sits at bits 4p..4p+3 and element 2p+1 at bits 16+4p..16+4p+3.
//
// Blocks are ordered [expert][row tile][k-block]; a whole row tile is contiguous.
// The gate/up GEMM interleaves its rows: row 2i of tile rt is gate feature
// 64*rt + i and row 2i+1 is up feature 64*rt + i, so one tile holds matching
// gate and up rows for 64 intermediate features.
//
// Activations feeding the tensor core as the B operand (expert-sorted hidden
// states and the intermediate activations, both fp16) are "blocked": [k-block][row
// group of 16 rows][16 rows x 128 bytes], each 128-byte row holding 64 fp16 reduction
// elements with the 16-byte chunks XOR-swizzled by (row % 8). A contiguous run of
// row groups of one k-block is exactly the shared-memory image the tensor core
// reads with a 128-byte-swizzle K-major descriptor.
#pragma once
#include <cstdint>

namespace moe {

constexpr int kGroup = 32;          // INT4 scale group along the reduction dimension
constexpr int kBM = 128;            // weight rows per tile (MMA M)
constexpr int kBK = 64;             // reduction elements per k-block
constexpr int kWBlockBytes = 4608;  // one packed (row tile, k-block) block
constexpr int kWCodeBytes = 4096;
constexpr int kBNMax = 64;          // largest token tile (MMA N)
constexpr int kRowGroup = 16;       // token rows per blocked row group
constexpr int kRowGroupBytes = kRowGroup * 128;
constexpr int kSmallTiles = 32;     // token tiles of a batch of at most 32 routed slots (one per expert)
constexpr int kSmallPadRows = 32 + 32 * (kRowGroup - 1);  // their padded rows (16 per expert at most)
constexpr int kMaxCtas = 256;       // persistent grid limit (tickets / scratch slots)
constexpr int kMaxExperts = 1024;

// Activation rows of the small-batch CUDA-core products ("step rows"): per padded
// row p and pipeline step kb (128 reduction elements) of an operand with KBn
// steps, 288 bytes at (p * KBn + kb) * 288. A row's steps are contiguous, so one
// copy brings several steps of a row. Each scale group g (32 elements) of the
// step is stored as 16-bit block fixed point: v = round(x * 2^e_g) with e_g
// chosen so that the group's largest |x| times 2^e_g lies in [2^13, 2^14)
// (xv_group_exp; 0 for an all-zero group):
//   bytes [64 g, 64 g + 64):  the group's four words of 8 elements, 16 bytes each,
//                             element i of a word in 16-bit slot kXvSlot[i]
//   bytes [256 + 8 g, +4):    2^-(e_g + 2) as a float (the factor 4 goes with the
//                             codes times 4 that the product kernels take)
//   bytes [260 + 8 g, +4):    32 times the sum of the group's 32 values (int32)
// The slot order pairs the values with the packed codes for dp2a: masking bits
// 2..5 of every byte of a packed word (of the word rotated right by 4) gives the
// codes of elements 2, 4, 3, 5 (0, 7, 1, 6), times 4, as bytes, which meet
// slots 0..3 (4..7).
constexpr int kXvStepBytes = 288;
__host__ __device__ constexpr int xv_slot(int i) {
  return i == 0 ? 4 : i == 1 ? 6 : i == 2 ? 0 : i == 3 ? 2 : i == 4 ? 1 : i == 5 ? 3 : i == 6 ? 7 : 5;
}
constexpr int kXvMaxExp = 100;  // |e_g| bound (2^-e_g stays a normal float)
#ifdef __CUDACC__
// e_g of a group whose largest magnitude is m (finite, >= 0).
__device__ __forceinline__ int xv_group_exp(float m) {
  if (!(m > 0.0f)) return 0;
  const int lg = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127;  // floor(log2 m) (normal m)
  const int e = 13 - lg;
  return e < -kXvMaxExp ? -kXvMaxExp : (e > kXvMaxExp ? kXvMaxExp : e);
}
// 16-bit value of x in a group with exponent e.
__device__ __forceinline__ int xv_quantize(float x, int e) {
  return __float2int_rn(x * __int_as_float((127 + e) << 23));
}
// Write group g's header into the step row at `row`.
__device__ __forceinline__ void xv_header(uint8_t* row, int g, int sum, int e) {
  int2 h;
  h.x = (125 - e) << 23;  // 2^-(e + 2): |e| <= kXvMaxExp, a normal float
  h.y = 32 * sum;         // |sum| < 2^19
  *reinterpret_cast<int2*>(row + 256 + 8 * g) = h;
}
#endif

// Byte offset of 16-bit element (row, k) inside one 16-row group of a k-block
// (row in [0, 16), k in [0, 64)).
__host__ __device__ __forceinline__ uint32_t blocked_offset(int row, int k) {
  return static_cast<uint32_t>(row * 128 + ((((k >> 3) ^ (row & 7)) & 7) << 4) + ((k & 7) << 1));
}

// One entry of the token-tile list built by the align kernel.
struct TokenTile {
  int expert;   // expert id
  int g0;       // first row group (16 rows) in the expert-sorted order
  int ngroups;  // row groups in the tile (MMA N = 16 * ngroups)
  int first;    // index of this expert's first token tile
};

// One tile of the CUDA-core (matrix-vector) products: up to kGemvRows routed rows
// of one expert -- padded rows p0 .. p0+n-1 of the expert-sorted order -- and the
// flat slot of each.
constexpr int kGemvRows = 4;
constexpr int kGemvMaxSlots = 256;      // routed slots up to which a forward may use them
constexpr int kGemvDefaultSlots = 256;  // ... and by default (measured faster than the tensor cores there)
struct GemvTile {
  int e, p0, n, pad;
  int slot[kGemvRows];
};

// Header words at the start of the workspace.
// kHdrSched: bit w set when the align kernel wrote cost-weighted stream-K
// boundaries for GEMM w (0 gate/up, 1 down; the general path only), clear for an
// even split of that GEMM's steps.
// kHdrNumGemvTiles: tiles in the CUDA-core tile list (written by the align kernel
// when the forward runs its products on the CUDA cores).
enum { kHdrStatus = 0, kHdrNumPadded = 1, kHdrNumTiles = 2, kHdrSched = 3, kHdrNumGemvTiles = 4, kHdrWords = 64 };

// Device status bits (the public values are in the C header).
enum {
  kStatusBadId = 1,       // a routed expert id outside [0, E) was skipped
  kStatusTimeout = 2,     // a pipeline wait gave up
  kStatusHSaturated = 4,  // an intermediate activation exceeded fp16's range (saturated)
  kStatusCheck = 8,       // self-checking build: a range check failed
  kStatusBadSched = 16    // malformed stream-K boundaries: the GEMMs split their steps evenly
};

// Per-token power-of-two prescale of the hidden states. A token row x is fed to
// the tensor cores as x * 2^-e (exact), with e chosen from the row's largest
// magnitude so that it lands in [4, 8): every row then sits in the same, safe
// part of fp16's range whatever its own scale. The gate/up epilogue multiplies
// the accumulators back by 2^e before SiLU and stores h * 2^-2e; the down
// epilogue multiplies by 2^2e. |e| <= kMaxRowExp keeps 2^e and 2^2e normal floats.
constexpr int kMaxRowExp = 63;
constexpr int kPadRowExp = -1000;  // the exponent recorded for a padding row
__host__ __device__ __forceinline__ float exp2_int(int e) {  // 2^e, |e| <= 126
#ifdef __CUDA_ARCH__
  return __int_as_float((127 + e) << 23);
#else
  union { int i; float f; } u;
  u.i = (127 + e) << 23;
  return u.f;
#endif
}

// Expert parallelism: a handle may hold only experts [e_begin, e_begin + E) of a
// layer with E_total experts (E_total == E, e_begin == 0 otherwise). A routed
// slot's expert id v maps to the local expert v - e_begin, or to -1 (skipped)
// when another part of the layer holds it; an id outside [0, E_total) is no
// expert of the layer at all: skipped too, and *bad is set.
__host__ __device__ __forceinline__ int local_expert(int v, int e_begin, int E, int E_total, bool* bad) {
  if (v < 0 || v >= E_total) {
    *bad = true;
    return -1;
  }
  const int l = v - e_begin;
  return (l >= 0 && l < E) ? l : -1;
}

// Relative cost of one pipeline step of a unit whose token tile holds ng row
// groups: a base of 8 plus `per_group` for every row group beyond the second. The
// weight stream (9 KB a step from HBM) and its conversion are the same for every
// tile; the activation copy from L2 is 4 KB per row group a step, which costs
// nothing extra while the weight stream sets the pace and starts to, alongside
// the larger MMAs and epilogue, at three and four row groups.
__host__ __device__ __forceinline__ int step_cost(int ng, int per_group) {
  return 8 + per_group * (ng > 2 ? ng - 2 : 0);
}

}  // namespace moe
