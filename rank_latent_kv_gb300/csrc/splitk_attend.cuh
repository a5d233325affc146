// Split-K single-token decode attention over fp16 K/V tiles in shared memory.
//
// The per-tile core shared by the dense fp16 comparator (K/V copied as they
// are) and the KIVI comparator (K/V dequantized from 2-bit codes into the
// same tiles): four warps, each owning 16 tokens of a 64-token tile; scores
// and weighted sums on the tensor cores (m16n8k16, fp32 accumulate) with the
// up-to-8 query heads of one KV head as the n8 side; online softmax in base 2.
// Tiles are [64 tokens][128 channels] fp16, 256 bytes a row, 16-byte chunks
// XOR-swizzled by the row so ldmatrix reads are conflict-free.
#pragma once

#include "palu_internal.cuh"

namespace palu {

constexpr int kSplitWarps = 4;
constexpr int kSplitTile = 64;                              // tokens per tile (16 per warp)
constexpr int kSplitTileBytes = kSplitTile * kHeadDim * 2;  // 16 KB per tensor
constexpr int kSplitPartStride = 2 + kHeadDim;              // (max, sum, acc[128]) per head

// Programmatic dependent launch: wait for the preceding launch's results /
// let the next launch be scheduled.  Both are no-ops without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float ex2f_(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory address of 16-byte chunk `ch` (0..15) of tile row `row`.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int ch) {
  return base + row * 256 + ((ch ^ (row & 7)) << 4);
}

// Running softmax state of one warp: rows g and g+8 of the n8 tile are heads
// 2c and 2c+1 (c = lane & 3); acc[mt] holds channels 16 mt .. 16 mt + 15.
struct SplitState {
  float m_run[2], l_run[2];
  float acc[8][4];
};

__device__ __forceinline__ void split_init(SplitState& st) {
  st.m_run[0] = st.m_run[1] = -INFINITY;
  st.l_run[0] = st.l_run[1] = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) st.acc[mt][0] = st.acc[mt][1] = st.acc[mt][2] = st.acc[mt][3] = 0.f;
}

// q of head g (lane >> 2) as the B operand (k = channel, n = head): a register
// pair for each 16-wide channel step; heads >= Gq are zero.
__device__ __forceinline__ void split_load_q(uint32_t qb[8][2], const __half* qh, bool valid, int c) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    if (valid) {
      qb[ks][0] = *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 2 * c);
      qb[ks][1] = *reinterpret_cast<const uint32_t*>(qh + 16 * ks + 8 + 2 * c);
    } else {
      qb[ks][0] = qb[ks][1] = 0u;
    }
  }
}

// The online softmax and weighted sum of one warp's 16 tokens, given their
// scores in base-2 units (sc[0..1]: token r0 + g, heads 2c and 2c+1;
// sc[2..3]: token r0 + g + 8; -inf for tokens that do not count).  The V rows
// of the tile at vst must be finite.
__device__ __forceinline__ void split_softmax_pv(SplitState& st, float sc[4], uint32_t vst, int r0, int lane) {
  const int mat = lane >> 3, rr = lane & 7;
  float bm0 = fmaxf(sc[0], sc[2]), bm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
  }
  const float mn0 = fmaxf(st.m_run[0], bm0), mn1 = fmaxf(st.m_run[1], bm1);
  if (mn0 != -INFINITY && mn1 != -INFINITY) {
    const float al0 = ex2f_(st.m_run[0] - mn0), al1 = ex2f_(st.m_run[1] - mn1);
    st.m_run[0] = mn0;
    st.m_run[1] = mn1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= al0;
      st.acc[mt][1] *= al1;
      st.acc[mt][2] *= al0;
      st.acc[mt][3] *= al1;
    }
    st.l_run[0] *= al0;
    st.l_run[1] *= al1;
    const float p0 = ex2f_(sc[0] - mn0), p1 = ex2f_(sc[1] - mn1), p2 = ex2f_(sc[2] - mn0), p3 = ex2f_(sc[3] - mn1);
    st.l_run[0] += p0 + p2;
    st.l_run[1] += p1 + p3;
    const uint32_t b0 = movmatrix_t(pack_f16x2(p0, p1));
    const uint32_t b1 = movmatrix_t(pack_f16x2(p2, p3));
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      // A = V^T (d x tokens) from the V rows: matrices (d0-7,t0-7), (d8-15,t0-7), (d0-7,t8-15), (d8-15,t8-15)
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(a0, a1, a2, a3, swz(vst, r0 + rr + ((mat >> 1) << 3), 2 * mt + (mat & 1)));
      mma_f16(st.acc[mt], a0, a1, a2, a3, b0, b1);
    }
  }
}

// One warp's 16 tokens (rows r0 .. r0+15 of the tile at kst / vst; token
// index of row r0 is tok0): scores, mask of tokens >= t1, online softmax and
// the weighted sum of the V rows.  Rows past t1 must hold finite values.
__device__ __forceinline__ void split_tile(SplitState& st, const uint32_t qb[8][2], uint32_t kst, uint32_t vst,
                                           int r0, int lane, long long tok0, long long t1, float scale_log2) {
  const int g = lane >> 2, mat = lane >> 3, rr = lane & 7;
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    // A = K rows (tokens x d): matrices (t0-7,d0-7), (t8-15,d0-7), (t0-7,d8-15), (t8-15,d8-15)
    uint32_t a0, a1, a2, a3;
    ldsm_x4(a0, a1, a2, a3, swz(kst, r0 + rr + ((mat & 1) << 3), 2 * ks + (mat >> 1)));
    mma_f16(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
  }
  // mask tokens past the end, scale to base 2
  const bool v0 = tok0 + g < t1, v1 = tok0 + g + 8 < t1;
  sc[0] = v0 ? sc[0] * scale_log2 : -INFINITY;
  sc[1] = v0 ? sc[1] * scale_log2 : -INFINITY;
  sc[2] = v1 ? sc[2] * scale_log2 : -INFINITY;
  sc[3] = v1 ? sc[3] * scale_log2 : -INFINITY;
  split_softmax_pv(st, sc, vst, r0, lane);
}

// Merge the warps' states (fixed warp order) and write the CTA's partial
// (max, sum, acc[128]) for each of the Gq heads.  merge is shared scratch.
__device__ __forceinline__ void split_write_partial(SplitState& st, float (*merge)[8][kSplitPartStride], int warp,
                                                    int lane, int Gq, float* part) {
  const int tid = threadIdx.x, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    st.l_run[0] += __shfl_xor_sync(0xffffffffu, st.l_run[0], x);
    st.l_run[1] += __shfl_xor_sync(0xffffffffu, st.l_run[1], x);
  }
  if (g == 0) {
    merge[warp][2 * c][0] = st.m_run[0];
    merge[warp][2 * c][1] = st.l_run[0];
    merge[warp][2 * c + 1][0] = st.m_run[1];
    merge[warp][2 * c + 1][1] = st.l_run[1];
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) merge[warp][2 * c + (e & 1)][2 + 16 * mt + g + 8 * (e >> 1)] = st.acc[mt][e];
  __syncthreads();
  for (int i = tid; i < Gq * kSplitPartStride; i += blockDim.x) {
    const int h = i / kSplitPartStride, e = i % kSplitPartStride;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSplitWarps; ++w) M = fmaxf(M, merge[w][h][0]);
    float o;
    if (e == 0) {
      o = M;
    } else {
      o = 0.f;
#pragma unroll
      for (int w = 0; w < kSplitWarps; ++w)
        if (merge[w][h][0] != -INFINITY) o += merge[w][h][e] * ex2f_(merge[w][h][0] - M);
    }
    part[i] = o;
  }
}

// An empty chunk's partial: max -inf, everything else 0.
__device__ __forceinline__ void split_write_empty(int Gq, float* part) {
  for (int i = threadIdx.x; i < Gq * kSplitPartStride; i += blockDim.x)
    part[i] = (i % kSplitPartStride) == 0 ? -INFINITY : 0.f;
}

// Merge the n_chunks partials of every (batch, KV head) stream into the
// output [batch, Hq, 128] (fp32 or fp16).  ws is [batch][Hkv][n_chunks][Gq][2+128].
palu_status split_combine(const float* ws, long long batch, int Hq, int Hkv, int n_chunks, void* out, int out_fp32,
                          cudaStream_t stream);

}  // namespace palu
