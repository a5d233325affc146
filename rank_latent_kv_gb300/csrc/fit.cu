// Basis fit of one tensor (K or V) of one layer.
//
// Method (page "PALU — True Low-Rank Latent Storage for Keys and Values",
// "How it works", prefill steps 1-3): split the KV heads into contiguous
// groups, stack each group's heads along the token axis, take a truncated SVD
// of the mean-centred rows -> shared basis V_g (D x r) and mean mu_g; the rank
// is explicit or set by an energy threshold, and one rank (the minimum over
// groups) is kept for all groups.
//
// The right singular vectors of X_c are the eigenvectors of the centred Gram
// matrix X_c^T X_c = X^T X - n mu mu^T.  GB300 plan:
//   1. gram_kernel: X^T X and the column sums of row chunks on tensor cores,
//      three CTAs per chunk for the symmetric 64 x 64 blocks (0,0), (0,1),
//      (1,1) (prefills above 64K rows per group; smaller ones use
//      gram_exact_kernel, exact accumulation on CUDA cores, because at small
//      row counts the rounding of each product sum is not yet averaged down).
//      fp16 operands are exact; each 64-row stage's product sum is promoted
//      from its fresh fp32 accumulator into an error-free fp32 pair, so the
//      chunk sums carry ~48-bit accuracy.  Rows are staged through swizzled
//      shared memory by cp.async.
//   2. gram_reduce_kernel: chunk partials summed in fp64, centred in fp64.
//   3. jacobi_kernel: one CTA per group (one launch for all the groups of
//      all tensors in a batch) diagonalises the 128x128 matrix with
//      parallel-ordered cyclic Jacobi rotations (64 disjoint pairs per round),
//      A as symmetric fp32 float pairs (about 48 significant bits; error-free
//      updates on the fp32 pipes), rotation angles in double-float and the
//      rotations accumulated in fp32, all in shared memory; then eigenvalues
//      sorted descending and each direction's sign fixed so its
//      largest-magnitude entry is positive.
//   4. host: energy-threshold rank per group, r = minimum.
#include <math.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "palu_internal.cuh"

namespace palu {

constexpr int kGramTile = 64;     // rows per shared-memory stage
constexpr int kGramStages = 3;
constexpr int kGramThreads = 256;

struct GramParams {
  const __half* x;
  float* part;      // [n_g][n_chunks][2][128][128]  (hi, lo)
  float* colpart;   // [n_g][n_chunks][2][128]
  long long seq, rows_g, chunk_rows;
  int Hkv, hg, n_chunks;
};

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(sz) : "memory");
}

// smem tile: 64 rows x 128 halves (256 B per row); 16-byte chunk ch of row r is
// stored at chunk (ch ^ (r & 7)) so ldmatrix row gathers are conflict-free.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int ch) {
  return base + row * 256 + ((ch ^ (row & 7)) << 4);
}

// grid (chunks, groups, 3): CTA z computes the 64 x 64 block (rb, cb) of the
// chunk's X^T X with (rb, cb) = (0, 0), (0, 1), (1, 1) for z = 0, 1, 2 (the
// matrix is symmetric: block (1, 0) is written as the transpose of (0, 1)),
// and the CTAs of the diagonal blocks the column sums of their 64 features.
// Rows stream through a 3-stage cp.async ring (only the 16-byte chunks of
// the features a block needs).  8 warps of 32 x 16 C each.
__global__ void __launch_bounds__(kGramThreads) gram_kernel(const GramParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, c4 = lane & 3;
  const int chunk = blockIdx.x, grp = blockIdx.y, z = blockIdx.z;
  const int rb = z == 2 ? 1 : 0, cb = z == 0 ? 0 : 1;
  const long long R0 = (long long)chunk * p.chunk_rows;
  const long long R1 = min(R0 + p.chunk_rows, p.rows_g);
  const int n_tiles = (int)((R1 - R0 + kGramTile - 1) / kGramTile);
  const uint32_t sbase = smem_addr(smem);

  // This thread's copy slots: rows (tid >> 4) + 16 i of each tile, chunk
  // tid & 15.  Each row's (batch, head in group, token) position advances
  // by 64 rows a tile with carries, instead of a division per copy.
  constexpr int kRowsPer = (kGramTile * 16) / kGramThreads;
  const int ch = tid & 15;
  const bool want = z == 1 || (ch >> 3) == rb;  // a diagonal block reads its own 64 features
  int cb_[kRowsPer], ch_[kRowsPer], ct_[kRowsPer];  // batch, head in group, token of the slot's row
  const __half* src_[kRowsPer];                      // that row's 16-byte chunk in x
  auto row_ptr = [&](int i) {
    return p.x + (((long long)cb_[i] * p.Hkv + (long long)grp * p.hg + ch_[i]) * p.seq + ct_[i]) * kHeadDim + ch * 8;
  };
#pragma unroll
  for (int i = 0; i < kRowsPer; ++i) {
    const long long R = R0 + (tid >> 4) + 16 * i;
    const long long bh = R / p.seq;
    ct_[i] = (int)(R - bh * p.seq);
    cb_[i] = (int)(bh / p.hg);
    ch_[i] = (int)(bh - (long long)cb_[i] * p.hg);
    src_[i] = row_ptr(i);
  }
  auto load_tile = [&](int tile, int stage) {
#pragma unroll
    for (int i = 0; i < kRowsPer; ++i) {
      const int row = (tid >> 4) + 16 * i;
      const long long R = R0 + (long long)tile * kGramTile + row;
      const bool valid = R < R1;
      if (want) {
        uint8_t* dst = smem + stage * (kGramTile * 256) + row * 256 + ((ch ^ (row & 7)) << 4);
        cp_async16_zfill(dst, valid ? src_[i] : p.x, valid);
      }
      // advance the slot's row by one tile: 64 rows further in the same
      // (batch, head) unless the token index passes the sequence's end
      ct_[i] += kGramTile;
      if (ct_[i] < p.seq) {
        src_[i] += kGramTile * kHeadDim;
      } else {
        do {
          ct_[i] -= (int)p.seq;
          if (++ch_[i] == p.hg) {
            ch_[i] = 0;
            ++cb_[i];
          }
        } while (ct_[i] >= p.seq);
        src_[i] = row_ptr(i);
      }
    }
  };

  const int wm = warp >> 2, wn = warp & 3;
  const int mbase = 64 * rb + 32 * wm, nbase = 64 * cb + 16 * wn;  // this warp's C rows / columns
  // Each stage's 64-row product sum (four chained 16-row MMAs) starts from a
  // zero accumulator and is then added into an unevaluated fp32 pair (hi, lo)
  // with an error-free sum: the rounding left is that of one 64-term product
  // sum, a random walk of sqrt(4) times a 16-term sum's; long fp32
  // accumulation chains would lose the ~1e-9 relative accuracy the trailing
  // retained directions of a decaying spectrum need.
  float Ch[2][2][4], Cl[2][2][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) Ch[a][b][e] = Cl[a][b][e] = 0.f;
  float Sh[2][4], Sl[2][4];  // column sums: X^T * ones (warps with wn == 0 of a diagonal block)
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int e = 0; e < 4; ++e) Sh[a][e] = Sl[a][e] = 0.f;
  const bool sums = z != 1 && wn == 0;
  const uint32_t ones = (g8 == 0) ? 0x3C003C00u : 0u;  // B[k][n] = 1 for n = 0

#pragma unroll
  for (int s = 0; s < kGramStages - 1; ++s) {
    if (s < n_tiles) load_tile(s, s);
    cp_async_commit();
  }
  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_async_wait<kGramStages - 2>();
    __syncthreads();
    const int nxt = tile + kGramStages - 1;
    if (nxt < n_tiles) load_tile(nxt, nxt % kGramStages);
    cp_async_commit();
    const uint32_t st = sbase + (tile % kGramStages) * (kGramTile * 256);
    const int mat = lane >> 3, rr = lane & 7;
    float T[2][2][4], U[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        T[a][0][e] = T[a][1][e] = 0.f;
        U[a][e] = 0.f;
      }
#pragma unroll
    for (int ks = 0; ks < kGramTile / 16; ++ks) {
      const int k0 = 16 * ks;
      uint32_t A[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int m0 = mbase + 16 * mi;
        // matrices: (k0-7, m0-7), (k0-7, m8-15), (k8-15, m0-7), (k8-15, m8-15)
        const int row = k0 + rr + ((mat >> 1) << 3);
        const int ch = (m0 >> 3) + (mat & 1);
        ldsm_x4_t(A[mi][0], A[mi][1], A[mi][2], A[mi][3], tile_addr(st, row, ch));
      }
      uint32_t Bf[2][2];
      {
        // matrices: (k0-7, n0-7), (k8-15, n0-7), (k0-7, n8-15), (k8-15, n8-15)
        const int row = k0 + rr + ((mat & 1) << 3);
        const int ch = (nbase >> 3) + (mat >> 1);
        ldsm_x4_t(Bf[0][0], Bf[0][1], Bf[1][0], Bf[1][1], tile_addr(st, row, ch));
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mma_f16(T[mi][nt], A[mi][0], A[mi][1], A[mi][2], A[mi][3], Bf[nt][0], Bf[nt][1]);
        if (sums) mma_f16(U[mi], A[mi][0], A[mi][1], A[mi][2], A[mi][3], ones, ones);
      }
    }
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float sm, err;
          two_sum(Ch[mi][nt][e], T[mi][nt][e], sm, err);
          Ch[mi][nt][e] = sm;
          Cl[mi][nt][e] = __fadd_rn(Cl[mi][nt][e], err);
        }
      if (sums)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float sm, err;
          two_sum(Sh[mi][e], U[mi][e], sm, err);
          Sh[mi][e] = sm;
          Sl[mi][e] = __fadd_rn(Sl[mi][e], err);
        }
    }
  }
  cp_async_wait<0>();

  float* dst = p.part + ((size_t)grp * p.n_chunks + chunk) * 2 * kHeadDim * kHeadDim;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = mbase + 16 * mi + g8 + 8 * (e >> 1);
        const int n = nbase + 8 * nt + 2 * c4 + (e & 1);
        dst[m * kHeadDim + n] = Ch[mi][nt][e];
        dst[kHeadDim * kHeadDim + m * kHeadDim + n] = Cl[mi][nt][e];
        if (z == 1) {  // the transposed block
          dst[n * kHeadDim + m] = Ch[mi][nt][e];
          dst[kHeadDim * kHeadDim + n * kHeadDim + m] = Cl[mi][nt][e];
        }
      }
  if (sums && c4 == 0) {
    float* cdst = p.colpart + ((size_t)grp * p.n_chunks + chunk) * 2 * kHeadDim;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      cdst[mbase + 16 * mi + g8] = Sh[mi][0];
      cdst[mbase + 16 * mi + g8 + 8] = Sh[mi][2];
      cdst[kHeadDim + mbase + 16 * mi + g8] = Sl[mi][0];
      cdst[kHeadDim + mbase + 16 * mi + g8 + 8] = Sl[mi][2];
    }
  }
}

// Exact Gram for small prefills: fp16 x fp16 products are exact in fp32 and
// are summed error-free into (hi, lo) pairs, so the chunk sums carry ~48-bit
// accuracy with no per-product-sum rounding.  Thread t owns the 8x8 block
// (t / 16, t % 16) of the 128x128 Gram; rows are staged as fp32 in shared
// memory, 64 at a time.  Same output layout as gram_kernel.
constexpr long long kExactGramRows = 65536;  // rows per group up to which this path is used

__global__ void __launch_bounds__(256) gram_exact_kernel(const GramParams p) {
  __shared__ __align__(16) float xs[kGramTile][kHeadDim + 4];
  const int tid = threadIdx.x, chunk = blockIdx.x, grp = blockIdx.y;
  const long long R0 = (long long)chunk * p.chunk_rows;
  const long long R1 = min(R0 + p.chunk_rows, p.rows_g);
  const int bi = tid >> 4, bj = tid & 15;
  float H[8][8], L[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) H[a][b] = L[a][b] = 0.f;
  float sh = 0.f, sl = 0.f;  // column sum of column tid (tid < 128)
  for (long long base = R0; base < R1; base += kGramTile) {
    const int nrows = (int)min((long long)kGramTile, R1 - base);
    __syncthreads();
    for (int i = tid; i < kGramTile * (kHeadDim / 8); i += 256) {
      const int row = i / (kHeadDim / 8), q = i % (kHeadDim / 8);
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (row < nrows) {
        const long long R = base + row;
        const long long bb = R / ((long long)p.hg * p.seq);
        const long long rem = R % ((long long)p.hg * p.seq);
        const long long hh = rem / p.seq, t = rem % p.seq;
        const uint4 w = *reinterpret_cast<const uint4*>(
            p.x + ((bb * p.Hkv + (long long)grp * p.hg + hh) * p.seq + t) * kHeadDim + 8 * q);
        const __half2* h2 = reinterpret_cast<const __half2*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h2[e]);
          v[2 * e] = f.x;
          v[2 * e + 1] = f.y;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) xs[row][8 * q + e] = v[e];
    }
    __syncthreads();
    for (int r = 0; r < nrows; ++r) {
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[r][8 * bi]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[r][8 * bi + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&xs[r][8 * bj]);
      const float4 b1 = *reinterpret_cast<const float4*>(&xs[r][8 * bj + 4]);
      const float xa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float xb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          float s, e;
          two_sum(H[a][b], __fmul_rn(xa[a], xb[b]), s, e);  // the product is exact
          H[a][b] = s;
          L[a][b] = __fadd_rn(L[a][b], e);
        }
      if (tid < kHeadDim) {
        float s, e;
        two_sum(sh, xs[r][tid], s, e);
        sh = s;
        sl = __fadd_rn(sl, e);
      }
    }
  }
  float* dst = p.part + ((size_t)grp * p.n_chunks + chunk) * 2 * kHeadDim * kHeadDim;
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int m = 8 * bi + a, n = 8 * bj + b;
      dst[m * kHeadDim + n] = H[a][b];
      dst[kHeadDim * kHeadDim + m * kHeadDim + n] = L[a][b];
    }
  if (tid < kHeadDim) {
    float* cdst = p.colpart + ((size_t)grp * p.n_chunks + chunk) * 2 * kHeadDim;
    cdst[tid] = sh;
    cdst[kHeadDim + tid] = sl;
  }
}

// grid (64, n_g), 256 threads: G[i][j] = sum_c (hi + lo) - colsum_i colsum_j / n, in fp64
__global__ void gram_reduce_kernel(const float* __restrict__ part, const float* __restrict__ colpart, int n_chunks,
                                   double n_rows, double* G, float* mu) {
  const int grp = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  const int i = e / kHeadDim, j = e % kHeadDim;
  const float* pp = part + (size_t)grp * n_chunks * 2 * kHeadDim * kHeadDim;
  const float* cp = colpart + (size_t)grp * n_chunks * 2 * kHeadDim;
  double s = 0.0, si = 0.0, sj = 0.0;
  for (int c = 0; c < n_chunks; ++c) {
    const float* pc = pp + (size_t)c * 2 * kHeadDim * kHeadDim;
    const float* cc = cp + (size_t)c * 2 * kHeadDim;
    s += (double)pc[e] + (double)pc[kHeadDim * kHeadDim + e];
    si += (double)cc[i] + (double)cc[kHeadDim + i];
    sj += (double)cc[j] + (double)cc[kHeadDim + j];
  }
  G[(size_t)grp * kHeadDim * kHeadDim + e] = s - si * sj / n_rows;
  if (i == 0) mu[(size_t)grp * kHeadDim + j] = (float)(sj / n_rows);
}

constexpr int kJacThreads = 544;  // 17 warps: a round's 2080 blocks in four passes
constexpr int kLdA = kHeadDim + 1;  // padded rows (fp64 and fp32)
constexpr int kMaxSweeps = 40;
// Rotate a pair while |a_pq| > max(kJacRel sqrt|a_pp a_qq|, kJacFloor ||A||_F):
// a few hundred units of the float pairs' rounding (2^-48)
constexpr double kJacRel = 1e-13;
constexpr double kJacFloor = 1e-14;

// Pairs of round `rnd` (0..126) of the round-robin (circle) ordering of 128 indices.
__device__ __forceinline__ void rr_pair(int rnd, int i, int& p, int& q) {
  const int n1 = kHeadDim - 1;
  if (i == 0) {
    p = rnd;
    q = n1;
  } else {
    p = (rnd + i) % n1;
    q = (rnd - i + n1) % n1;
  }
  if (p > q) {
    const int t = p;
    p = q;
    q = t;
  }
}

// The matrix being diagonalised is held as float pairs (hi + lo, about 48
// significant bits): every rotation update runs on the fp32 pipes with
// error-free transformations, where this part's fp64 rate would make it the
// fit's bottleneck.  A product of two pairs, unnormalised (p + e):
__device__ __forceinline__ void df_prod(float ah, float al, float bh, float bl, float& p, float& e) {
  p = __fmul_rn(ah, bh);
  e = __fmaf_rn(ah, bh, -p);
  e = __fmaf_rn(ah, bl, e);
  e = __fmaf_rn(al, bh, e);
}
// (p1 + e1) + (p2 + e2) as a normalised pair
__device__ __forceinline__ void df_sum(float p1, float e1, float p2, float e2, float& hi, float& lo) {
  float s, err;
  two_sum(p1, p2, s, err);
  const float t = __fadd_rn(__fadd_rn(e1, e2), err);
  hi = __fadd_rn(s, t);
  lo = __fsub_rn(t, __fsub_rn(hi, s));
}
// (x, y) <- (c x - s y, s x + c y) for pairs x, y and rotation (c, s)
__device__ __forceinline__ void df_rotate(float ch, float cl, float sh, float sl, float& xh, float& xl, float& yh,
                                          float& yl) {
  float p1, e1, p2, e2, nxh, nxl, nyh, nyl;
  df_prod(ch, cl, xh, xl, p1, e1);
  df_prod(-sh, -sl, yh, yl, p2, e2);
  df_sum(p1, e1, p2, e2, nxh, nxl);
  df_prod(sh, sl, xh, xl, p1, e1);
  df_prod(ch, cl, yh, yl, p2, e2);
  df_sum(p1, e1, p2, e2, nyh, nyl);
  xh = nxh;
  xl = nxl;
  yh = nyh;
  yl = nyl;
}

// Double-float (fp32 pair) arithmetic for the rotation angles (Dekker's
// error-free product and sum; the pair division and square root refine an
// fp32 quotient or root by the residual): about 44 significant bits, on the
// fp32 pipes, where this part's fp64 rate made the angles the slow step of a
// round.  Explicit rounding intrinsics keep the compiler from contracting
// the error terms.
struct Dfl {
  float h, l;
};
__device__ __forceinline__ Dfl dfl_norm(float s, float e) {  // |s| >= |e|
  const float h = __fadd_rn(s, e);
  return Dfl{h, __fsub_rn(e, __fsub_rn(h, s))};
}
__device__ __forceinline__ Dfl dfl_neg(Dfl a) { return Dfl{-a.h, -a.l}; }
__device__ __forceinline__ Dfl dfl_add(Dfl a, Dfl b) {  // operands that do not cancel
  float s, e;
  two_sum(a.h, b.h, s, e);
  return dfl_norm(s, __fadd_rn(__fadd_rn(e, a.l), b.l));
}
__device__ __forceinline__ Dfl dfl_add_exact(Dfl a, Dfl b) {  // also under cancellation
  float s1, e1, s2, e2;
  two_sum(a.h, b.h, s1, e1);
  two_sum(a.l, b.l, s2, e2);
  const Dfl t = dfl_norm(s1, __fadd_rn(e1, s2));
  return dfl_norm(t.h, __fadd_rn(t.l, e2));
}
__device__ __forceinline__ Dfl dfl_mul(Dfl a, Dfl b) {
  const float p = __fmul_rn(a.h, b.h);
  float e = __fmaf_rn(a.h, b.h, -p);
  e = __fmaf_rn(a.h, b.l, e);
  e = __fmaf_rn(a.l, b.h, e);
  return dfl_norm(p, e);
}
__device__ __forceinline__ Dfl dfl_div(Dfl a, Dfl b) {
  const float q1 = __fdiv_rn(a.h, b.h);
  const Dfl r1 = dfl_add_exact(a, dfl_neg(dfl_mul(Dfl{q1, 0.f}, b)));
  const float q2 = __fdiv_rn(r1.h, b.h);
  const Dfl r2 = dfl_add_exact(r1, dfl_neg(dfl_mul(Dfl{q2, 0.f}, b)));
  const float q3 = __fdiv_rn(r2.h, b.h);
  return dfl_add(dfl_norm(q1, q2), Dfl{q3, 0.f});
}
__device__ __forceinline__ Dfl dfl_sqrt(Dfl a) {  // a > 0
  const float s1 = __fsqrt_rn(a.h);
  const float p = __fmul_rn(s1, s1), pe = __fmaf_rn(s1, s1, -p);  // s1^2 = p + pe exactly
  const Dfl r = dfl_add_exact(a, Dfl{-p, -pe});
  return dfl_norm(s1, __fdiv_rn(r.h, __fmul_rn(2.f, s1)));
}

constexpr int kJacBlocks = 64 * 65 / 2;  // 2x2 blocks (pair a, pair b), a <= b, of a round

// A is kept symmetric: entry {i, j} lives once, at row min(i, j), column
// max(i, j) of the padded array.
__device__ __forceinline__ int sym(int i, int j) { return i < j ? i * kLdA + j : j * kLdA + i; }

// The matrices of one Jacobi launch: CTA i diagonalises matrix i (a head
// group of one fitted tensor) and writes its sorted basis and eigenvalues.
constexpr int kMaxJacBatch = 256;
struct JacMatrix {
  const double* G;        // [128][128] centred Gram matrix
  float* basis;           // [128][128]
  double* eigvals;        // [128]
  unsigned int* err;      // the tensor's device error word
};
struct JacBatch {
  JacMatrix m[kMaxJacBatch];
};

__global__ void __launch_bounds__(kJacThreads) jacobi_kernel(const __grid_constant__ JacBatch jb) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* Ah = reinterpret_cast<float*>(smem);                     // [128][129] high parts (upper triangle)
  float* Al = Ah + kHeadDim * kLdA;                                // [128][129] low parts
  float* V = Al + kHeadDim * kLdA;                                 // [128][129]
  float* rot = V + kHeadDim * kLdA;                                // [2][4][64]: c, s as pairs, two rounds
  int* pq = reinterpret_cast<int*>(rot + 2 * 4 * 64);              // [2][2][64]: p, q, two rounds
  int* cnt = pq + 2 * 2 * 64;                                      // rotations this sweep
  double* red = reinterpret_cast<double*>(cnt + 4);                // [kJacThreads / 32]
  int* order = reinterpret_cast<int*>(red + kJacThreads / 32);     // [128]
  uint16_t* blk = reinterpret_cast<uint16_t*>(order + kHeadDim);  // [kJacBlocks]: a * 64 + b
  auto a64 = [&](int i, int j) { return (double)Ah[sym(i, j)] + (double)Al[sym(i, j)]; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const JacMatrix& mat = jb.m[blockIdx.x];
  const double* Gg = mat.G;
  double fro = 0.0;
  for (int e = tid; e < kHeadDim * kHeadDim; e += kJacThreads) {
    const int i = e / kHeadDim, j = e % kHeadDim;
    const double a = Gg[e];
    if (i <= j) {
      const float ah = (float)a;
      Ah[i * kLdA + j] = ah;
      Al[i * kLdA + j] = (float)(a - (double)ah);
    }
    V[i * kLdA + j] = (i == j) ? 1.f : 0.f;
    fro += a * a;
  }
  for (int a = tid; a < 64; a += kJacThreads) {
    const int base = a * 64 - a * (a - 1) / 2;  // blocks (a, a..63) start here
    for (int b = a; b < 64; ++b) blk[base + b - a] = (uint16_t)(a * 64 + b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) fro += __shfl_xor_sync(0xffffffffu, fro, o);
  if (lane == 0) red[warp] = fro;
  if (tid == 0) *cnt = 0;
  __syncthreads();
  double fro_all = 0.0;
  for (int w = 0; w < kJacThreads / 32; ++w) fro_all += red[w];
  // off-diagonal entries below these bounds are at the pairs' rounding level
  const double floor_abs = kJacFloor * sqrt(fro_all);

  // The rotations of round k (buffer k & 1) from the current A, by warps 0-1,
  // in double-float arithmetic: theta = (a_qq - a_pp) / (2 a_pq),
  // t = sign(theta) / (|theta| + sqrt(theta^2 + 1)) (1 / (2 theta) past
  // |theta| = 2^40), c = 1 / sqrt(t^2 + 1), s = t c.  The difference a_qq -
  // a_pp is formed exactly, so theta keeps its relative accuracy when the
  // diagonal entries nearly cancel.
  const float floor_f = (float)floor_abs;
  auto angles = [&](int rnd, int buf) {
    int p, q;
    rr_pair(rnd, tid, p, q);
    const Dfl apq{Ah[sym(p, q)], Al[sym(p, q)]}, app{Ah[p * kLdA + p], Al[p * kLdA + p]},
        aqq{Ah[q * kLdA + q], Al[q * kLdA + q]};
    Dfl c{1.f, 0.f}, s{0.f, 0.f};
    if (fabsf(apq.h) > fmaxf((float)kJacRel * sqrtf(fabsf(app.h)) * sqrtf(fabsf(aqq.h)), floor_f)) {
      const Dfl th = dfl_div(dfl_add_exact(aqq, dfl_neg(app)), Dfl{2.f * apq.h, 2.f * apq.l});
      Dfl t;
      if (fabsf(th.h) > 0x1p40f) {
        t = dfl_div(Dfl{0.5f, 0.f}, th);
      } else {
        const Dfl root = dfl_sqrt(dfl_add(dfl_mul(th, th), Dfl{1.f, 0.f}));
        t = dfl_div(Dfl{1.f, 0.f}, dfl_add(th.h >= 0.f ? th : dfl_neg(th), root));
        if (th.h < 0.f) t = dfl_neg(t);
      }
      c = dfl_div(Dfl{1.f, 0.f}, dfl_sqrt(dfl_add(dfl_mul(t, t), Dfl{1.f, 0.f})));
      s = dfl_mul(t, c);
      atomicAdd(cnt, 1);
    }
    float* r = rot + buf * 256;
    int* ix = pq + buf * 128;
    ix[tid] = p;
    ix[64 + tid] = q;
    r[tid] = c.h;
    r[64 + tid] = c.l;
    r[128 + tid] = s.h;
    r[192 + tid] = s.l;
  };
  // V <- V J for the rotations in buffer buf, by threads from t0 on
  auto rotate_v = [&](int buf, int t0) {
    const float* r = rot + buf * 256;
    const int* ix = pq + buf * 128;
    for (int e = tid - t0; e < 64 * kHeadDim; e += kJacThreads - t0) {
      const int i = e % 64, k = e / 64;
      const float sf = r[128 + i];
      if (sf != 0.f) {
        const int p = ix[i], q = ix[64 + i];
        const float cf = r[i];
        const float vp = V[k * kLdA + p], vq = V[k * kLdA + q];
        V[k * kLdA + p] = cf * vp - sf * vq;
        V[k * kLdA + q] = sf * vp + cf * vq;
      }
    }
  };

  if (tid < 64) angles(0, 0);
  __syncthreads();
  int sweep = 0, done = 0, gr = 0;  // gr: rounds so far (a sweep has an odd number), picks the buffer
  for (; sweep < kMaxSweeps && !done; ++sweep) {
    for (int rnd = 0; rnd < kHeadDim - 1; ++rnd, ++gr) {
      const int buf = gr & 1;
      const float* r = rot + buf * 256;
      const int* ix = pq + buf * 128;
      // A <- J^T A J block by block: rows of pair a by its rotation, then
      // columns of pair b by its rotation (the off-diagonal entry of a
      // rotated pair is annihilated and set to 0)
      for (int k = tid; k < kJacBlocks; k += kJacThreads) {
        const int a = blk[k] >> 6, b = blk[k] & 63;
        const bool ra = r[128 + a] != 0.f, rb = r[128 + b] != 0.f;
        if (!ra && !rb) continue;
        const int pa = ix[a], qa = ix[64 + a], pb = ix[b], qb = ix[64 + b];
        const float cah = r[a], cal = r[64 + a], sah = r[128 + a], sal = r[192 + a];
        if (a == b) {
          const int ipp = pa * kLdA + pa, ipq = sym(pa, qa), iqq = qa * kLdA + qa;
          float x00h = Ah[ipp], x00l = Al[ipp], x01h = Ah[ipq], x01l = Al[ipq], x11h = Ah[iqq], x11l = Al[iqq];
          float x10h = x01h, x10l = x01l;
          df_rotate(cah, cal, sah, sal, x00h, x00l, x10h, x10l);  // column p: rows p, q
          df_rotate(cah, cal, sah, sal, x01h, x01l, x11h, x11l);  // column q
          df_rotate(cah, cal, sah, sal, x00h, x00l, x01h, x01l);  // row p: columns p, q
          df_rotate(cah, cal, sah, sal, x10h, x10l, x11h, x11l);  // row q
          Ah[ipp] = x00h;
          Al[ipp] = x00l;
          Ah[iqq] = x11h;
          Al[iqq] = x11l;
          Ah[ipq] = 0.f;
          Al[ipq] = 0.f;
          continue;
        }
        const int i00 = sym(pa, pb), i01 = sym(pa, qb), i10 = sym(qa, pb), i11 = sym(qa, qb);
        float x00h = Ah[i00], x00l = Al[i00], x01h = Ah[i01], x01l = Al[i01];
        float x10h = Ah[i10], x10l = Al[i10], x11h = Ah[i11], x11l = Al[i11];
        if (ra) {
          df_rotate(cah, cal, sah, sal, x00h, x00l, x10h, x10l);
          df_rotate(cah, cal, sah, sal, x01h, x01l, x11h, x11l);
        }
        if (rb) {
          const float cbh = r[b], cbl = r[64 + b], sbh = r[128 + b], sbl = r[192 + b];
          df_rotate(cbh, cbl, sbh, sbl, x00h, x00l, x01h, x01l);
          df_rotate(cbh, cbl, sbh, sbl, x10h, x10l, x11h, x11l);
        }
        Ah[i00] = x00h;
        Al[i00] = x00l;
        Ah[i01] = x01h;
        Al[i01] = x01l;
        Ah[i10] = x10h;
        Al[i10] = x10l;
        Ah[i11] = x11h;
        Al[i11] = x11l;
      }
      __syncthreads();
      // next round's angles (warps 0-1) beside this round's V update (the rest)
      const bool last = rnd == kHeadDim - 2;
      if (last && tid == 0) {
        done = *cnt == 0;  // read by thread 0 only, shared below
        red[0] = done;
        *cnt = 0;
      }
      if (last) __syncthreads();
      if (last) done = red[0] != 0.0;
      if (tid < 64) {
        if (!(last && (done || sweep + 1 == kMaxSweeps))) angles(last ? 0 : rnd + 1, buf ^ 1);
      } else {
        rotate_v(buf, 64);
      }
      __syncthreads();
    }
  }
  if (tid == 0 && !done) atomicOr(mat.err, PALU_DEVERR_NOT_CONVERGED);

  // sort by descending eigenvalue (stable: ties keep index order)
  if (tid < kHeadDim) {
    const double li = a64(tid, tid);
    int pos = 0;
    for (int j = 0; j < kHeadDim; ++j) {
      const double lj = a64(j, j);
      pos += (lj > li) || (lj == li && j < tid);
    }
    order[pos] = tid;
  }
  __syncthreads();
  if (tid < kHeadDim) {
    const int src = order[tid];
    // canonical sign: largest-magnitude entry positive (first index among ties)
    int arg = 0;
    float best = -1.f;
    for (int d = 0; d < kHeadDim; ++d) {
      const float a = fabsf(V[d * kLdA + src]);
      if (a > best) {
        best = a;
        arg = d;
      }
    }
    const float sgn = V[arg * kLdA + src] < 0.f ? -1.f : 1.f;
    float* bg = mat.basis;
    for (int d = 0; d < kHeadDim; ++d) bg[d * kHeadDim + tid] = sgn * V[d * kLdA + src];
    mat.eigvals[tid] = fmax(a64(src, src), 0.0);
  }
}

static size_t jacobi_smem() {
  return 3 * sizeof(float) * kHeadDim * kLdA + sizeof(float) * 2 * 256 + sizeof(int) * 2 * 128 + sizeof(int) * 4 +
         sizeof(double) * (kJacThreads / 32) + sizeof(int) * kHeadDim + sizeof(uint16_t) * kJacBlocks;
}

struct FitLayout {
  int n_chunks;
  long long chunk_rows;
  size_t part_off, col_off, G_off, err_off, total;
};

// Rows per chunk, in whole 64-row tiles: enough chunks over all groups for
// one CTA per SM (the exact kernel), or for two CTAs per SM with three block
// CTAs per chunk (the tensor-core kernel).
static FitLayout fit_layout(int n_groups, long long rows_g) {
  FitLayout f;
  const long long sms = device_sm_count();
  const bool tc = rows_g > kExactGramRows;
  long long per = (rows_g * n_groups * (tc ? 3 : 1) + (tc ? 2 : 1) * sms - 1) / ((tc ? 2 : 1) * sms);
  per = (per + kGramTile - 1) / kGramTile * kGramTile;
  f.chunk_rows = std::max<long long>(kGramTile, std::min<long long>(1LL << 20, per));
  f.n_chunks = (int)((rows_g + f.chunk_rows - 1) / f.chunk_rows);
  f.part_off = 0;
  f.col_off = align_up(f.part_off + sizeof(float) * 2 * (size_t)n_groups * f.n_chunks * kHeadDim * kHeadDim, 256);
  f.G_off = align_up(f.col_off + sizeof(float) * 2 * (size_t)n_groups * f.n_chunks * kHeadDim, 256);
  f.err_off = align_up(f.G_off + sizeof(double) * (size_t)n_groups * kHeadDim * kHeadDim, 256);
  f.total = f.err_off + 256;
  return f;
}

// energy-threshold rank (same definition as the method's "retain 90% of
// singular value energy"; sigma or sigma^2 reading), clamped to [1, D]
static int energy_rank(const double* lam, int D, double tau, int mode) {
  std::vector<double> cum(D);
  double run = 0.0;
  for (int i = 0; i < D; ++i) {
    const double l = lam[i] > 0.0 ? lam[i] : 0.0;
    run += (mode == PALU_ENERGY_SIGMA) ? sqrt(l) : l;
    cum[i] = run;
  }
  const double total = cum[D - 1];
  if (!(total > 0.0)) return 1;
  for (int i = 0; i < D; ++i)
    if (cum[i] / total >= tau) return std::max(1, i + 1);
  return D;
}

static palu_status check_fit_args(const palu_config* cfg, int64_t batch, int32_t kv_heads, int64_t seq) {
  if (!cfg) return fail(PALU_ERR_INVALID_ARG, "config is NULL");
  if (cfg->head_dim != kHeadDim) return fail(PALU_ERR_UNSUPPORTED, "head_dim must be 128");
  if (cfg->n_head_groups < 1 || kv_heads < 1 || kv_heads % cfg->n_head_groups != 0)
    return fail(PALU_ERR_INVALID_ARG, "kv_heads must be a positive multiple of n_head_groups");
  if (batch < 1 || seq < 1) return fail(PALU_ERR_INVALID_ARG, "batch and seq must be >= 1");
  if (cfg->rank < 0) return fail(PALU_ERR_INVALID_ARG, "rank must be >= 0");
  if (cfg->rank == 0 && !(cfg->energy_threshold > 0.0 && cfg->energy_threshold <= 1.0))
    return fail(PALU_ERR_INVALID_ARG, "energy_threshold must be in (0, 1]");
  if (cfg->energy_mode != PALU_ENERGY_SIGMA && cfg->energy_mode != PALU_ENERGY_SIGMA2)
    return fail(PALU_ERR_INVALID_ARG, "energy_mode must be PALU_ENERGY_SIGMA or PALU_ENERGY_SIGMA2");
  const long long rows_g = batch * (long long)(kv_heads / cfg->n_head_groups) * seq;
  if (rows_g < 2) return fail(PALU_ERR_INVALID_ARG, "need at least 2 rows per head group");
  if (rows_g / kGramTile > 2147483647LL) return fail(PALU_ERR_UNSUPPORTED, "prefill too large");
  return PALU_OK;
}

}  // namespace palu

using namespace palu;

namespace palu {

// Gram matrix and mean of one tensor's head groups (prefill steps 1-2): the
// partial sums go to part / colpart (shared by the tensors of a batch, which
// run one after the other on the stream), the fp64 reduction to G and mu.
static palu_status launch_gram(const palu_config* cfg, const void* x, int64_t batch, int32_t kv_heads, int64_t seq,
                               const FitLayout& fl, uint8_t* part_ws, double* G, float* mu, cudaStream_t strm) {
  const int ng = cfg->n_head_groups;
  const int hg = kv_heads / ng;
  const long long rows_g = batch * (long long)hg * seq;
  GramParams gp;
  gp.x = static_cast<const __half*>(x);
  gp.part = reinterpret_cast<float*>(part_ws + fl.part_off);
  gp.colpart = reinterpret_cast<float*>(part_ws + fl.col_off);
  gp.seq = seq;
  gp.rows_g = rows_g;
  gp.Hkv = kv_heads;
  gp.hg = hg;
  gp.n_chunks = fl.n_chunks;
  gp.chunk_rows = fl.chunk_rows;
  palu_status st;
  if (rows_g <= kExactGramRows) {
    gram_exact_kernel<<<dim3(fl.n_chunks, ng), 256, 0, strm>>>(gp);
  } else {
    const int gram_smem = kGramStages * kGramTile * 256;
    int per_sm = 0;
    st = kernel_occupancy(reinterpret_cast<const void*>(gram_kernel), kGramThreads, gram_smem, &per_sm);
    if (st != PALU_OK) return st;
    gram_kernel<<<dim3(fl.n_chunks, ng, 3), kGramThreads, gram_smem, strm>>>(gp);
  }
  st = cuda_check(cudaGetLastError(), "gram_kernel launch");
  if (st != PALU_OK) return st;
  gram_reduce_kernel<<<dim3(kHeadDim * kHeadDim / 256, ng), 256, 0, strm>>>(gp.part, gp.colpart, fl.n_chunks,
                                                                             (double)rows_g, G, mu);
  return cuda_check(cudaGetLastError(), "gram_reduce_kernel launch");
}

// Diagonalise the listed matrices, kMaxJacBatch per launch (one CTA, one SM,
// each).
static palu_status launch_jacobi(const std::vector<JacMatrix>& mats, cudaStream_t strm) {
  const size_t jsm = jacobi_smem();
  int per_sm = 0;
  palu_status st = kernel_occupancy(reinterpret_cast<const void*>(jacobi_kernel), kJacThreads, (int)jsm, &per_sm);
  if (st != PALU_OK) return st;
  for (size_t i0 = 0; i0 < mats.size(); i0 += kMaxJacBatch) {
    JacBatch jb;
    std::memset(&jb, 0, sizeof(jb));
    const size_t n = std::min<size_t>(kMaxJacBatch, mats.size() - i0);
    for (size_t i = 0; i < n; ++i) jb.m[i] = mats[i0 + i];
    jacobi_kernel<<<(unsigned)n, kJacThreads, jsm, strm>>>(jb);
    st = cuda_check(cudaGetLastError(), "jacobi_kernel launch");
    if (st != PALU_OK) return st;
  }
  return PALU_OK;
}

// Workspace of a batch: one partial-sum area (the largest any tensor needs),
// then per tensor its Gram matrices and error word.
struct BatchLayout {
  size_t part_bytes;
  std::vector<FitLayout> fl;
  std::vector<size_t> g_off, err_off;
  size_t total;
};
static BatchLayout batch_layout(const palu_config* cfgs, int n, int64_t batch, int32_t kv_heads, int64_t seq) {
  BatchLayout b;
  b.part_bytes = 0;
  for (int t = 0; t < n; ++t) {
    const int ng = cfgs[t].n_head_groups;
    b.fl.push_back(fit_layout(ng, batch * (long long)(kv_heads / ng) * seq));
    b.part_bytes = std::max(b.part_bytes, b.fl.back().G_off);
  }
  size_t o = align_up(b.part_bytes, 256);
  for (int t = 0; t < n; ++t) {
    b.g_off.push_back(o);
    o = align_up(o + sizeof(double) * (size_t)cfgs[t].n_head_groups * kHeadDim * kHeadDim, 256);
    b.err_off.push_back(o);
    o += 256;
  }
  b.total = o;
  return b;
}

// Ranks from the eigenvalues (prefill step 3) once the stream has finished.
static palu_status finish_ranks(const palu_config* cfg, const std::vector<double>& lam, unsigned int herr,
                                int32_t* rank_out, int32_t* group_ranks) {
  if (herr) return fail(PALU_ERR_DEVICE, "eigen-solver did not converge within its sweep limit");
  int rmin = kHeadDim;
  for (int g = 0; g < cfg->n_head_groups; ++g) {
    const int rg = cfg->rank > 0 ? std::min(cfg->rank, kHeadDim)
                                 : energy_rank(lam.data() + (size_t)g * kHeadDim, kHeadDim, cfg->energy_threshold,
                                               cfg->energy_mode);
    if (group_ranks) group_ranks[g] = rg;
    rmin = std::min(rmin, rg);
  }
  *rank_out = rmin;
  return PALU_OK;
}

// Fit n tensors of equal shape: every tensor's Gram matrices first, then one
// Jacobi launch over all their head groups, then one synchronisation.
static palu_status fit_many(const palu_config* cfgs, int n, const void* const* xs, int64_t batch, int32_t kv_heads,
                            int64_t seq, void* workspace, size_t workspace_bytes, float* const* bases,
                            float* const* mus, double* const* eigvals, int32_t* ranks_out, int32_t* group_ranks,
                            void* stream) {
  if (n < 1) return fail(PALU_ERR_INVALID_ARG, "n_tensors must be >= 1");
  if (!cfgs || !xs || !bases || !mus || !eigvals || !ranks_out)
    return fail(PALU_ERR_INVALID_ARG, "configs, x, basis, mu, eigvals and rank_out arrays must be non-NULL");
  for (int t = 0; t < n; ++t) {
    palu_status st = check_fit_args(&cfgs[t], batch, kv_heads, seq);
    if (st != PALU_OK) return st;
    if (!xs[t] || !bases[t] || !mus[t] || !eigvals[t])
      return fail(PALU_ERR_INVALID_ARG, "x, basis, mu and eigvals must be non-NULL for every tensor");
    if ((uintptr_t)xs[t] & 15) return fail(PALU_ERR_INVALID_ARG, "x must be 16-byte aligned");
  }
  if (!workspace || ((uintptr_t)workspace & 255))
    return fail(PALU_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  const BatchLayout bl = batch_layout(cfgs, n, batch, kv_heads, seq);
  if (workspace_bytes < bl.total)
    return fail(PALU_ERR_INVALID_ARG, "fit workspace too small: need " + std::to_string(bl.total) + " bytes");
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  std::vector<JacMatrix> mats;
  for (int t = 0; t < n; ++t) {
    unsigned int* err = reinterpret_cast<unsigned int*>(ws + bl.err_off[t]);
    palu_status st = cuda_check(cudaMemsetAsync(err, 0, sizeof(unsigned int), strm), "memset");
    if (st != PALU_OK) return st;
    double* G = reinterpret_cast<double*>(ws + bl.g_off[t]);
    st = launch_gram(&cfgs[t], xs[t], batch, kv_heads, seq, bl.fl[t], ws, G, mus[t], strm);
    if (st != PALU_OK) return st;
    for (int g = 0; g < cfgs[t].n_head_groups; ++g)
      mats.push_back(JacMatrix{G + (size_t)g * kHeadDim * kHeadDim, bases[t] + (size_t)g * kHeadDim * kHeadDim,
                               eigvals[t] + (size_t)g * kHeadDim, err});
  }
  palu_status st = launch_jacobi(mats, strm);
  if (st != PALU_OK) return st;
  std::vector<std::vector<double>> lam(n);
  std::vector<unsigned int> herr(n, 0u);
  for (int t = 0; t < n; ++t) {
    lam[t].resize((size_t)cfgs[t].n_head_groups * kHeadDim);
    st = cuda_check(cudaMemcpyAsync(lam[t].data(), eigvals[t], sizeof(double) * lam[t].size(), cudaMemcpyDeviceToHost,
                                    strm),
                    "copy eigenvalues");
    if (st != PALU_OK) return st;
    st = cuda_check(cudaMemcpyAsync(&herr[t], ws + bl.err_off[t], sizeof(unsigned int), cudaMemcpyDeviceToHost, strm),
                    "copy error word");
    if (st != PALU_OK) return st;
  }
  st = cuda_check(cudaStreamSynchronize(strm), "cudaStreamSynchronize(fit)");
  if (st != PALU_OK) return st;
  size_t goff = 0;
  for (int t = 0; t < n; ++t) {
    st = finish_ranks(&cfgs[t], lam[t], herr[t], &ranks_out[t], group_ranks ? group_ranks + goff : nullptr);
    if (st != PALU_OK) return st;
    goff += cfgs[t].n_head_groups;
  }
  return PALU_OK;
}

}  // namespace palu

extern "C" palu_status palu_fit_workspace_size(const palu_config* cfg, int64_t batch, int32_t kv_heads, int64_t seq,
                                               size_t* bytes) {
  palu_status st = check_fit_args(cfg, batch, kv_heads, seq);
  if (st != PALU_OK) return st;
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = batch_layout(cfg, 1, batch, kv_heads, seq).total;
  return PALU_OK;
}

extern "C" palu_status palu_fit(const palu_config* cfg, const void* x, int64_t batch, int32_t kv_heads, int64_t seq,
                                void* workspace, size_t workspace_bytes, float* basis, float* mu, double* eigvals,
                                int32_t* rank_out, int32_t* group_ranks, void* stream) {
  if (!cfg) return fail(PALU_ERR_INVALID_ARG, "config is NULL");
  return fit_many(cfg, 1, &x, batch, kv_heads, seq, workspace, workspace_bytes, &basis, &mu, &eigvals, rank_out,
                  group_ranks, stream);
}

extern "C" palu_status palu_fit_batch_workspace_size(const palu_config* cfgs, int32_t n_tensors, int64_t batch,
                                                     int32_t kv_heads, int64_t seq, size_t* bytes) {
  if (!cfgs || n_tensors < 1) return fail(PALU_ERR_INVALID_ARG, "configs must be non-NULL and n_tensors >= 1");
  for (int t = 0; t < n_tensors; ++t) {
    palu_status st = check_fit_args(&cfgs[t], batch, kv_heads, seq);
    if (st != PALU_OK) return st;
  }
  if (!bytes) return fail(PALU_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = batch_layout(cfgs, n_tensors, batch, kv_heads, seq).total;
  return PALU_OK;
}

extern "C" palu_status palu_fit_batch(const palu_config* cfgs, int32_t n_tensors, const void* const* x, int64_t batch,
                                      int32_t kv_heads, int64_t seq, void* workspace, size_t workspace_bytes,
                                      float* const* basis, float* const* mu, double* const* eigvals,
                                      int32_t* rank_out, int32_t* group_ranks, void* stream) {
  return fit_many(cfgs, n_tensors, x, batch, kv_heads, seq, workspace, workspace_bytes, basis, mu, eigvals, rank_out,
                  group_ranks, stream);
}
