// Internal definitions shared by the host API and the kernels of the library.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gmmfr {

// ---------------------------------------------------------------- tiling constants
constexpr int kTileN = 128;                // output columns per weight tile = MMA M
constexpr int kTileK = 128;                // K bytes per pipeline stage (4 MMAs of K = 32)
constexpr int kWTileBytes = kTileN * kTileK;  // 16 KB of FP8 weights per tile
constexpr int kSfChunk = 512;              // scale bytes of a 128-row x 4-block tile
constexpr int kPrepTileBytes = kWTileBytes + kSfChunk;  // 16896: prepared tile = weights + scales
// Packed E2M1 x E2M1 (kind::mxf4): the same 128-byte rows hold 256 K elements (two per
// byte), so a stage carries 4 MMAs of K = 64 and 8 scales per row (two scale chunks).
constexpr int kTileK4 = 256;                              // K elements per FP4 stage
constexpr int kPrepTileBytes4 = kWTileBytes + 2 * kSfChunk;  // 17408
constexpr int kTokBox = 16;                // token rows per TMA box
// warp 0 TMA, 1 MMA, 2..5 epilogue, then the token-scale packers: one for FP8 operands, two
// for packed E2M1 (eight scale words per lane per stage)
__host__ __device__ constexpr int gemm_threads(bool fp4) { return fp4 ? 256 : 224; }
constexpr int kMaxExperts = 1024;

// Workspace header: word 0 = number of error slots written by the last GEMM
// launch, words 1..kMaxErrSlots = each CTA's device error bits.
constexpr int kMaxErrSlots = 1023;
constexpr int kHdrBytes = 4096;

constexpr uint32_t kErrBadGroupList = 1u;
constexpr uint32_t kErrBadRowIndex = 2u;
constexpr uint32_t kErrTimeout = 4u;
constexpr uint32_t kErrBadExpertId = 8u;

struct PrepParams {
  const uint8_t* x2;
  const uint8_t* scale;
  uint8_t* prepared;
  int64_t E, K, N;
  int32_t NT, KB, Ks;
  int32_t transpose_x2;
  int32_t scale_per_expert;
  int32_t fp4;         // x2 holds packed E2M1 codes
  int32_t fp4_native;  // with fp4: keep them packed (256-K tiles for kind::mxf4), else expand to E4M3
};
cudaError_t launch_expand_fp4(const uint8_t* packed, uint8_t* fp8, int64_t n_bytes, cudaStream_t s);
// x1 [M, K] (packed E2M1 with fp4) -> [M, Kp] bytes, Kp = K rounded up to 16, zero past K
cudaError_t launch_pad_tokens(const uint8_t* x1, uint8_t* dst, int64_t M, int64_t K, int64_t Kp, bool fp4,
                              cudaStream_t s);

struct GemmParams {
  const uint8_t* prepared;
  const int64_t* group_list;
  const uint8_t* pertoken_scale;  // [M, 2*Ks]
  const float* logit;
  const void* row_index;
  const uint16_t* shared;  // bf16 bits; added here only in atomic mode
  const uint16_t* bias;    // [E, N] bf16 bits or null
  float* out;
  float* ybuf;             // deterministic: [split][M][N]
  // deterministic: tokens of each out row (CSR, unordered within a row), built by CTA 0
  int32_t* csr_cnt;        // [batch] counts
  int32_t* csr_row_ptr;    // [batch + 1]
  int32_t* csr_cursor;     // [batch] scatter cursors
  int32_t* csr_sorted;     // [M] token indices grouped by row
  uint32_t* hdr;           // error slots (see kHdrBytes)
  int64_t M, N, K, batch;
  int64_t shared_rows, shared_offset;
  float shared_weight;
  int32_t E, group_list_type;
  int32_t NT, KB, Ks;
  int32_t split;           // deterministic K split count
  int32_t deterministic;
  int32_t row_i32;
  int32_t tmax_fixed;      // 0: token group width chosen on the device from the largest expert
  int32_t fp4;             // packed E2M1 tokens and weights: 256-K stages, kind::mxf4 MMAs
  uint32_t idesc;          // instruction descriptor without N and scale-factor ids
  int64_t timeout_ns;
  int32_t test_stall;      // testing aid: wait on a barrier nothing arrives on
  int32_t reverse_units;   // testing aid (deterministic mode): each CTA walks its units last to first
};

struct CombineParams {
  const int32_t* row_ptr;
  const int32_t* sorted;
  const float* ybuf;
  const uint16_t* shared;
  float* out;
  int64_t M, N, batch;
  int64_t shared_rows, shared_offset;
  float shared_weight;
  int32_t split;
};

// MoE routing step (kernels_route.cu)
struct RouteScatterParams {
  const void* topk_ids;          // [M] int64 or int32
  const float* topk_weights;     // [M] or null
  const uint8_t* x;              // [batch, K]
  const uint8_t* x_scale;        // [batch, 2*Ks]
  uint8_t* x1;                   // [M, K]
  uint8_t* pertoken_scale;       // [M, 2*Ks]
  int64_t* group_list;           // [E]
  int64_t* row_index;            // [M]
  float* logit;                  // [M] or null
  int32_t* perm;                 // [M] or null
  int32_t* rank;                 // workspace [M]: stable rank of an entry within its tile and key
  int32_t* tile_counts;          // workspace [tiles][E+1]: counts, then each tile's first position per key
  uint32_t* hdr;                 // error words
  int64_t M, K, topk;
  int32_t E, Ks, ids_i32, group_list_type, vec16;
};
cudaError_t launch_route_kernels(const RouteScatterParams& p, cudaStream_t s);

// Grouped SwiGLU expert FFN (kernels_ffn.cu)
struct FfnPrepParams {
  const uint16_t* w13;  // [E*H, 2I] bf16
  const uint16_t* w2;   // [E*I, H] bf16
  uint8_t* prepared;
  int64_t H, I;
  int32_t E, NT1, KB1, NT2, KB2;
};
struct FfnParams {
  const uint8_t* prepared;  // tiles of this GEMM
  const int32_t* cumsum;    // [E+1]
  __nv_bfloat16* out;       // GEMM1: sw [N, I]; GEMM2: result [N, H]
  uint32_t* hdr;
  int64_t N;
  int64_t out_cols;         // I (GEMM1) or H (GEMM2)
  int32_t E, NT, KB;
  int32_t gate_up;          // 1: SwiGLU epilogue
  int32_t slot_base;        // first error slot of this launch
  int32_t dependent;        // launched as a programmatic dependent of GEMM1: sw is read only after
                            // griddepcontrol.wait (weight tiles stream before it)
  uint32_t idesc;
  int64_t timeout_ns;
};
struct TokenMaps;
cudaError_t launch_ffn_prep(const FfnPrepParams& p, cudaStream_t s);
cudaError_t launch_ffn_gemm(const TokenMaps& tmaps, const FfnParams& p, int grid, cudaStream_t s);

// launchers (defined next to their kernels)
cudaError_t launch_prep(const PrepParams& p, cudaStream_t s);
// x1 [M, K] as 2-D tensors of 128-byte rows, boxes of 16, 32, 64 and 128 rows (128-byte swizzle).
struct TokenMaps {
  CUtensorMap m[4];
};
cudaError_t launch_gemm(const TokenMaps& tmaps, const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);
int gemm_smem_bytes();
}  // namespace gmmfr

#include "gmmfr.h"
namespace gmmfr {
gmmfr_status record_error(gmmfr_status st, const char* message);

}  // namespace gmmfr
