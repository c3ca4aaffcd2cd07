// Memory-bound kernels of the Muon step: momentum with the Frobenius norm,
// scale + cast + orientation of the Newton-Schulz input, and the scaled
// weight update (or the copy-out of the orthogonalised matrix).
//
// The pages fix only that Muon keeps optimizer state ("lower memory than
// AdamW", "How to train a GPT model in 3 minutes", section 2) and steps the
// hidden matrices with an orthogonalised update. The momentum form
// buf <- beta*buf + g with the Nesterov look-ahead u = g + beta*buf, the
// normalisation X0 = u / (||u||_F + eps), the orientation rule (transpose when
// rows > cols) and the update W <- W - lr * max(1, rows/cols)^0.5 * O are the
// stated configuration of this path.
//
// All kernels take a table of matrices as a __grid_constant__ parameter and
// map blocks to matrices by a prefix of per-matrix block counts, so one launch
// serves a whole batch of mixed shapes. Global accesses are 16-byte vectors
// whenever alignment allows.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace muon {

constexpr int kEwThreads = 256;
constexpr int kFlatChunk = 8192;  // elements per block in the flat kernels (4 vectors of 8 per thread)
constexpr int kTile = 64;         // transpose tile edge
constexpr int kEwMax = 128;       // matrices per launch

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint16_t f_to_bf16(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

template <bool kF32>
__device__ __forceinline__ void store8(void* base, int64_t idx, const float (&v)[8]) {
  if (kF32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
      w[h] = static_cast<uint32_t>(f_to_bf16(v[2 * h])) | (static_cast<uint32_t>(f_to_bf16(v[2 * h + 1])) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// x held as a pair of bf16 values (precise carry): hi = bf16(x), lo = bf16(x - hi), so that hi + lo
// keeps about 16 significant bits of x.
__device__ __forceinline__ uint16_t lo_part(float x, uint16_t hi) { return f_to_bf16(x - bf16_to_f(hi)); }

// Stores eight values as bf16 at hi + idx and, when lo is not null, their low parts at lo + idx.
__device__ __forceinline__ void store8_split(uint16_t* hi, uint16_t* lo, int64_t idx, const float (&v)[8]) {
  uint32_t wh[4], wl[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint16_t h0 = f_to_bf16(v[2 * h]), h1 = f_to_bf16(v[2 * h + 1]);
    wh[h] = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
    wl[h] = static_cast<uint32_t>(lo_part(v[2 * h], h0)) | (static_cast<uint32_t>(lo_part(v[2 * h + 1], h1)) << 16);
  }
  *reinterpret_cast<uint4*>(hi + idx) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  if (lo) *reinterpret_cast<uint4*>(lo + idx) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
}

__device__ __forceinline__ void store1_split(uint16_t* hi, uint16_t* lo, int64_t idx, float v) {
  const uint16_t h = f_to_bf16(v);
  hi[idx] = h;
  if (lo) lo[idx] = lo_part(v, h);
}

// Eight consecutive elements in their storage form (one or two 16-byte words), so that every
// load of a thread can be in flight before any of them is unpacked.
template <bool kF32>
struct Raw8 {
  uint4 w[kF32 ? 2 : 1];
};

template <bool kF32>
__device__ __forceinline__ Raw8<kF32> ld_raw8(const void* base, int64_t idx) {
  Raw8<kF32> r;
  if constexpr (kF32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + idx);
    r.w[0] = p[0];
    r.w[1] = p[1];
  } else {
    r.w[0] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx);
  }
  return r;
}

template <bool kF32>
__device__ __forceinline__ void unpack8(const Raw8<kF32>& r, float (&v)[8]) {
  if constexpr (kF32) {
    v[0] = __uint_as_float(r.w[0].x); v[1] = __uint_as_float(r.w[0].y);
    v[2] = __uint_as_float(r.w[0].z); v[3] = __uint_as_float(r.w[0].w);
    v[4] = __uint_as_float(r.w[1].x); v[5] = __uint_as_float(r.w[1].y);
    v[6] = __uint_as_float(r.w[1].z); v[7] = __uint_as_float(r.w[1].w);
  } else {
    const uint32_t ww[4] = {r.w[0].x, r.w[0].y, r.w[0].z, r.w[0].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[2 * h] = __uint_as_float(ww[h] << 16);
      v[2 * h + 1] = __uint_as_float(ww[h] & 0xFFFF0000u);
    }
  }
}

template <bool kF32>
__device__ __forceinline__ float load1(const void* base, int64_t idx) {
  return kF32 ? static_cast<const float*>(base)[idx] : bf16_to_f(static_cast<const uint16_t*>(base)[idx]);
}

template <bool kF32>
__device__ __forceinline__ void store1(void* base, int64_t idx, float v) {
  if (kF32)
    static_cast<float*>(base)[idx] = v;
  else
    static_cast<uint16_t*>(base)[idx] = f_to_bf16(v);
}

// Index of the matrix whose block range holds block b (block_begin ascending).
template <typename Mat>
__device__ __forceinline__ int owner_of_block(const Mat* m, int count, int b) {
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (m[mid].block_begin <= b)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  return s;
}

// ---------------------------------------------------------------------------
// K4a: momentum (+ Nesterov) and the per-matrix sum of squares of u.
// kStep = false skips the momentum and takes u = g: the norm pass of
// muon_orthogonalize.
// ---------------------------------------------------------------------------

struct MomMat {
  const void* g;       // gradient or orthogonalize input (fp32 or bf16)
  float* buf;          // momentum, fp32
  uint16_t* u;         // bf16 u in the Newton-Schulz orientation (n x m, ld_u), or nullptr (norm only)
  uint16_t* u_lo;      // its low parts (precise carry), same layout, or nullptr
  int64_t ld_g, ld_buf, ld_u;
  int rows, cols;      // caller orientation
  int transposed;      // u = (g-side matrix)^T: written through a 128 x 64 shared-memory tile
  int tiles_c;         // transposed: tiles along the caller's columns
  int vec_ok;          // 16-byte vectors: flat path needs ld == cols everywhere and cols % 8 == 0;
                       // transposed path needs every ld % 8 == 0; both need aligned pointers
  int block_begin;     // first block of this matrix in the launch
  int nchunks;         // blocks of this matrix = partial sums
  float* partial;      // nchunks partial sums of u^2
  int* ticket;         // arrivals; zero between calls (the last block resets it)
  float* inv;          // out: 1 / (||u||_F + eps)
  float* post;         // out (or nullptr): scale the first Newton-Schulz products apply to u (1 when
                       // the norm is outside the fold range and u was scaled in place instead)
};

struct MomArgs {
  MomMat m[kEwMax];
  int count;
  float beta;
  int nesterov;
  float eps;
  int force_rescale;   // 1: every matrix takes the in-place scale (no folded scale)
};

// Norms for which the unscaled u can go through the fp32-accumulated Gram safely: every
// element is below 1e10 (no overflow of its products) and typical elements are far above the
// square root of the smallest normal float (no underflow). Outside it u is scaled first.
constexpr float kFoldMinNorm = 1e-10f, kFoldMaxNorm = 1e10f;

template <bool kStep, bool kSrcF32>
__device__ __forceinline__ float momentum_u(float g, float& b, float beta, int nesterov) {
  if (!kStep) return g;
  const float nb = beta * b + g;
  b = nb;
  return nesterov ? g + beta * nb : nb;
}

template <bool kStep, bool kSrcF32>
__global__ void __launch_bounds__(kEwThreads, kSrcF32 ? 3 : 4) momentum_norm_kernel(const __grid_constant__ MomArgs a) {
  grid_dependency_wait();
  const int j = owner_of_block(a.m, a.count, static_cast<int>(blockIdx.x));
  const MomMat& M = a.m[j];
  const int chunk = static_cast<int>(blockIdx.x) - M.block_begin;
  const float beta = a.beta;
  float ss = 0.f;

  if (!M.transposed) {
    const int64_t cols = M.cols;
    const int64_t n = static_cast<int64_t>(M.rows) * cols;
    const int64_t e0 = static_cast<int64_t>(chunk) * kFlatChunk;
    const int64_t e1 = min(n, e0 + kFlatChunk);
    if (M.vec_ok) {
      // Contiguous rows on every side (ld == cols), so element e sits at offset e.
      constexpr int V = kFlatChunk / (kEwThreads * 8);
      Raw8<kSrcF32> gr[V];
      Raw8<true> br[V];
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = e0 + (static_cast<int64_t>(v) * kEwThreads + threadIdx.x) * 8;
        if (e < e1) {
          gr[v] = ld_raw8<kSrcF32>(M.g, e);
          if (kStep) br[v] = ld_raw8<true>(M.buf, e);
        }
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = e0 + (static_cast<int64_t>(v) * kEwThreads + threadIdx.x) * 8;
        if (e < e1) {
          float g[8], b[8], u[8];
          unpack8<kSrcF32>(gr[v], g);
          if (kStep) unpack8<true>(br[v], b);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            u[k] = momentum_u<kStep, kSrcF32>(g[k], b[k], beta, a.nesterov);
            ss += u[k] * u[k];
          }
          if (kStep) store8<true>(M.buf, e, b);
          if (M.u) store8_split(M.u, M.u_lo, e, u);
        }
      }
    } else {
      for (int64_t e = e0 + threadIdx.x; e < e1; e += kEwThreads) {
        const int64_t row = e / cols, col = e - row * cols;
        const float g = load1<kSrcF32>(M.g, row * M.ld_g + col);
        float b = kStep ? M.buf[row * M.ld_buf + col] : 0.f;
        const float u = momentum_u<kStep, kSrcF32>(g, b, beta, a.nesterov);
        if (kStep) M.buf[row * M.ld_buf + col] = b;
        if (M.u) store1_split(M.u, M.u_lo, row * M.ld_u + col, u);
        ss += u * u;
      }
    }
  } else {
    // Caller tile rows r0..r0+127, columns c0..c0+63; u^T rows c0..c0+63, columns r0..r0+127.
    __shared__ float tile[128][kTile + 1];
    const int r0 = (chunk / M.tiles_c) * 128;
    const int c0 = (chunk % M.tiles_c) * kTile;
    const int sub = threadIdx.x >> 3;
    const int c8 = (threadIdx.x & 7) * 8;
    constexpr int P1 = 128 / 32;
    Raw8<kSrcF32> gr[P1];
    Raw8<true> br[P1];
#pragma unroll
    for (int p = 0; p < P1; ++p) {
      const int gr_ = r0 + p * 32 + sub, gc = c0 + c8;
      if (M.vec_ok && gr_ < M.rows && gc + 7 < M.cols) {
        gr[p] = ld_raw8<kSrcF32>(M.g, static_cast<int64_t>(gr_) * M.ld_g + gc);
        if (kStep) br[p] = ld_raw8<true>(M.buf, static_cast<int64_t>(gr_) * M.ld_buf + gc);
      }
    }
#pragma unroll
    for (int p = 0; p < P1; ++p) {
      const int r = p * 32 + sub;
      const int row = r0 + r, gc = c0 + c8;
      float u[8];
      if (M.vec_ok && row < M.rows && gc + 7 < M.cols) {
        float g[8], b[8];
        unpack8<kSrcF32>(gr[p], g);
        if (kStep) unpack8<true>(br[p], b);
#pragma unroll
        for (int k = 0; k < 8; ++k) u[k] = momentum_u<kStep, kSrcF32>(g[k], b[k], beta, a.nesterov);
        if (kStep) store8<true>(M.buf, static_cast<int64_t>(row) * M.ld_buf + gc, b);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          u[k] = 0.f;
          if (row < M.rows && gc + k < M.cols) {
            const float g = load1<kSrcF32>(M.g, static_cast<int64_t>(row) * M.ld_g + gc + k);
            float b = kStep ? M.buf[static_cast<int64_t>(row) * M.ld_buf + gc + k] : 0.f;
            u[k] = momentum_u<kStep, kSrcF32>(g, b, beta, a.nesterov);
            if (kStep) M.buf[static_cast<int64_t>(row) * M.ld_buf + gc + k] = b;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ss += u[k] * u[k];
        tile[r][c8 + k] = u[k];
      }
    }
    if (M.u) {
      __syncthreads();
      // 16 threads per u^T row (128 columns), 16 rows per pass.
      const int drow = threadIdx.x >> 4;
      const int dcol = (threadIdx.x & 15) * 8;
#pragma unroll
      for (int p = 0; p < kTile / 16; ++p) {
        const int cc = p * 16 + drow;
        const int dr = c0 + cc, dc = r0 + dcol;
        if (dr >= M.cols) continue;
        float uv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) uv[k] = tile[dcol + k][cc];
        const int64_t di = static_cast<int64_t>(dr) * M.ld_u + dc;
        if (M.vec_ok && dc + 7 < M.rows) {
          store8_split(M.u, M.u_lo, di, uv);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (dc + k < M.rows) store1_split(M.u, M.u_lo, di + k, uv[k]);
        }
      }
    }
  }

  // Deterministic norm: every block stores its partial, the last block to
  // arrive sums the partials in index order.
  __shared__ float wsum[kEwThreads / 32];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ss = warp_sum(ss);
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kEwThreads / 32; ++w) s += wsum[w];
    M.partial[chunk] = s;
    __threadfence();
    const int t = atomicAdd(M.ticket, 1);
    is_last = (t == M.nchunks - 1);
  }
  __syncthreads();
  if (is_last) {
    __threadfence();
    float s = 0.f;
    for (int i = threadIdx.x; i < M.nchunks; i += kEwThreads) s += __ldcg(M.partial + i);
    s = warp_sum(s);
    __syncthreads();
    if (lane == 0) wsum[warp] = s;
    __syncthreads();
    __shared__ float inv_s;
    __shared__ int fold_s;
    if (threadIdx.x == 0) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kEwThreads / 32; ++w) tot += wsum[w];
      const float norm = sqrtf(tot);
      const float inv = 1.0f / (norm + a.eps);
      *M.inv = inv;
      const bool fold = !a.force_rescale && norm >= kFoldMinNorm && norm <= kFoldMaxNorm;
      if (M.post) *M.post = fold ? inv : 1.0f;
      inv_s = inv;
      fold_s = fold ? 1 : 0;
      *M.ticket = 0;
    }
    __syncthreads();
    if (M.u && !fold_s) {
      // Norm outside the fold range: this block scales the whole of u in place (rare; every other
      // block's u is visible after its fence and ticket).
      const float f = inv_s;
      const int64_t n = M.transposed ? M.cols : M.rows, m = M.transposed ? M.rows : M.cols;
      for (int64_t e = threadIdx.x; e < n * m; e += kEwThreads) {
        const int64_t row = e / m, col = e - row * m, i = row * M.ld_u + col;
        float x = bf16_to_f(__ldcg(M.u + i));
        if (M.u_lo) x += bf16_to_f(__ldcg(M.u_lo + i));
        store1_split(M.u, M.u_lo, i, x * f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// K1 / K4b / copy-out: dst (optionally transposed) = f(src).
//   kScale : dst(bf16) = src * inv                  (X0 from u or the input)
//   kUpdate: dst -= scale * src                     (W <- W - lr*s*O)
//   kCopy  : dst = src                              (O to the caller's buffer)
// With transposed != 0 the destination is sc x sr and dst(c, r) = f(src(r, c)),
// done through a 64 x 64 shared-memory tile so both sides stay coalesced.
// ---------------------------------------------------------------------------

enum MapMode { kScale = 0, kUpdate = 1, kCopy = 2 };

struct MapMat {
  const void* src;
  void* dst;
  const uint16_t* src_lo;  // kUpdate / kCopy with the precise carry: low parts of src (bf16, src's layout)
  uint16_t* dst_lo;        // kScale with the precise carry: low parts of dst (bf16, dst's layout)
  int64_t ld_src, ld_dst;
  int sr, sc;          // source rows, cols
  int transposed;
  int vec_ok;          // 16-byte vectors allowed: flat path needs ld == cols on both sides,
                       // transposed path needs both lds % 8 == 0; both need 16-byte aligned pointers
  int block_begin;
  int tiles_c;         // transposed: tiles along the source columns
  float scale;         // kUpdate: lr * s
  const float* inv;    // kScale: device scalar
};

struct MapArgs {
  MapMat m[kEwMax];
  int count;
  float keep;  // kUpdate: 1 - lr * weight_decay, applied to the old destination
};

template <int kMode, bool kDstF32>
__device__ __forceinline__ void map_apply1(const MapMat& M, float f, float s, int64_t di, float keep) {
  if (kMode == kUpdate)
    store1<kDstF32>(M.dst, di, keep * load1<kDstF32>(M.dst, di) - f * s);
  else if (kMode == kScale && M.dst_lo)
    store1_split(static_cast<uint16_t*>(M.dst), M.dst_lo, di, s * f);
  else
    store1<kDstF32>(M.dst, di, (kMode == kScale) ? s * f : s);
}

// The source value at si: src, plus its low part under the precise carry.
template <bool kSrcF32>
__device__ __forceinline__ float map_src1(const MapMat& M, int64_t si) {
  float v = load1<kSrcF32>(M.src, si);
  if (M.src_lo) v += bf16_to_f(M.src_lo[si]);
  return v;
}

// Eight results at di: dst (and dst_lo for kScale under the precise carry).
template <int kMode, bool kDstF32>
__device__ __forceinline__ void map_store8(const MapMat& M, int64_t di, const float (&d)[8]) {
  if (kMode == kScale && !kDstF32)
    store8_split(static_cast<uint16_t*>(M.dst), M.dst_lo, di, d);
  else
    store8<kDstF32>(M.dst, di, d);
}

// d = f(s) for eight elements: the old destination values dold are used by kUpdate only.
template <int kMode>
__device__ __forceinline__ void map_combine8(float f, const float (&sv)[8], const float (&dold)[8], float (&d)[8],
                                             float keep) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (kMode == kUpdate)
      d[k] = keep * dold[k] - f * sv[k];
    else if (kMode == kScale)
      d[k] = sv[k] * f;
    else
      d[k] = sv[k];
  }
}

constexpr int kTileRows = 128;  // transposed path: source tile of 128 rows x 64 columns

template <int kMode, bool kSrcF32, bool kDstF32>
__global__ void __launch_bounds__(kEwThreads, 3) map_kernel(const __grid_constant__ MapArgs a) {
  grid_dependency_wait();
  const int j = owner_of_block(a.m, a.count, static_cast<int>(blockIdx.x));
  const MapMat& M = a.m[j];
  const int blk = static_cast<int>(blockIdx.x) - M.block_begin;
  const float f = (kMode == kScale) ? __ldg(M.inv) : M.scale;

  if (!M.transposed) {
    const int64_t cols = M.sc;
    const int64_t n = static_cast<int64_t>(M.sr) * cols;
    const int64_t e0 = static_cast<int64_t>(blk) * kFlatChunk;
    const int64_t e1 = min(n, e0 + kFlatChunk);
    if (M.vec_ok) {
      // Contiguous rows on both sides (ld == cols): element e sits at offset e.
      constexpr int V = kFlatChunk / (kEwThreads * 8);
      Raw8<kSrcF32> sr[V];
      Raw8<kDstF32> dr[V];
      Raw8<false> lr[V];
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = e0 + (static_cast<int64_t>(v) * kEwThreads + threadIdx.x) * 8;
        if (e < e1) {
          sr[v] = ld_raw8<kSrcF32>(M.src, e);
          if (kMode != kScale && M.src_lo) lr[v] = ld_raw8<false>(M.src_lo, e);
          if (kMode == kUpdate) dr[v] = ld_raw8<kDstF32>(M.dst, e);
        }
      }
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t e = e0 + (static_cast<int64_t>(v) * kEwThreads + threadIdx.x) * 8;
        if (e < e1) {
          float sv[8], dold[8], d[8];
          unpack8<kSrcF32>(sr[v], sv);
          if (kMode != kScale && M.src_lo) {
            float lo[8];
            unpack8<false>(lr[v], lo);
#pragma unroll
            for (int k = 0; k < 8; ++k) sv[k] += lo[k];
          }
          if (kMode == kUpdate) unpack8<kDstF32>(dr[v], dold);
          map_combine8<kMode>(f, sv, dold, d, a.keep);
          map_store8<kMode, kDstF32>(M, e, d);
        }
      }
    } else {
      for (int64_t e = e0 + threadIdx.x; e < e1; e += kEwThreads) {
        const int64_t row = e / cols, col = e - row * cols;
        map_apply1<kMode, kDstF32>(M, f, map_src1<kSrcF32>(M, row * M.ld_src + col), row * M.ld_dst + col, a.keep);
      }
    }
    return;
  }

  // Transposed: source tile rows r0..r0+127, columns c0..c0+63; destination rows c0..c0+63,
  // columns r0..r0+127. Both sides move 16-byte vectors along their own rows.
  __shared__ float tile[kTileRows][kTile + 1];
  const int r0 = (blk / M.tiles_c) * kTileRows;
  const int c0 = (blk % M.tiles_c) * kTile;
  // Phase 1 mapping: 8 threads per source row, 32 rows per pass.
  const int sub = threadIdx.x >> 3;
  const int c8 = (threadIdx.x & 7) * 8;
  // Phase 2 mapping: 16 threads per destination row (128 columns), 16 rows per pass.
  const int drow = threadIdx.x >> 4;
  const int dcol = (threadIdx.x & 15) * 8;
  constexpr int P1 = kTileRows / 32, P2 = kTile / 16;
  Raw8<kSrcF32> sraw[P1];
  Raw8<kDstF32> draw[P2];
  Raw8<false> lraw[P1];
#pragma unroll
  for (int p = 0; p < P1; ++p) {
    const int gr = r0 + p * 32 + sub, gc = c0 + c8;
    if (M.vec_ok && gr < M.sr && gc + 7 < M.sc) {
      sraw[p] = ld_raw8<kSrcF32>(M.src, static_cast<int64_t>(gr) * M.ld_src + gc);
      if (kMode != kScale && M.src_lo) lraw[p] = ld_raw8<false>(M.src_lo, static_cast<int64_t>(gr) * M.ld_src + gc);
    }
  }
  if (kMode == kUpdate) {
#pragma unroll
    for (int p = 0; p < P2; ++p) {
      const int dr = c0 + p * 16 + drow, dc = r0 + dcol;
      if (M.vec_ok && dr < M.sc && dc + 7 < M.sr) draw[p] = ld_raw8<kDstF32>(M.dst, static_cast<int64_t>(dr) * M.ld_dst + dc);
    }
  }
#pragma unroll
  for (int p = 0; p < P1; ++p) {
    const int r = p * 32 + sub;
    const int gr = r0 + r, gc = c0 + c8;
    float v[8];
    if (M.vec_ok && gr < M.sr && gc + 7 < M.sc) {
      unpack8<kSrcF32>(sraw[p], v);
      if (kMode != kScale && M.src_lo) {
        float lo[8];
        unpack8<false>(lraw[p], lo);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] += lo[k];
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        v[k] = (gr < M.sr && gc + k < M.sc) ? map_src1<kSrcF32>(M, static_cast<int64_t>(gr) * M.ld_src + gc + k) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[r][c8 + k] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < P2; ++p) {
    const int cc = p * 16 + drow;
    const int dr = c0 + cc, dc = r0 + dcol;
    if (dr >= M.sc) continue;
    float sv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) sv[k] = tile[dcol + k][cc];
    const int64_t di = static_cast<int64_t>(dr) * M.ld_dst + dc;
    if (M.vec_ok && dc + 7 < M.sr) {
      float dold[8], d[8];
      if (kMode == kUpdate) unpack8<kDstF32>(draw[p], dold);
      map_combine8<kMode>(f, sv, dold, d, a.keep);
      map_store8<kMode, kDstF32>(M, di, d);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (dc + k < M.sr) map_apply1<kMode, kDstF32>(M, f, sv[k], di + k, a.keep);
    }
  }
}

}  // namespace muon
