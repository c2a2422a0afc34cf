// S5 + S6: split-KV sparse flash-decode over the selected cells.
//
// llama.cpp issue #28734 ("decode slows linearly with context"), fix summary,
// lever1: flash attention runs over only the top-k K/V set, so the cost is
// O(top_k) instead of O(n_kv); sparse256: the head shape is DKQ = DV = 256
// with 8 query heads per KV head (ncols2 = 8).  The author's q8-compact
// follow-up keeps the sparse path for a q8_0 cache; here q8_0 rows are
// gathered as int8 + fp16 scales and dequantised in shared memory, so the
// whole cache is never converted (the O(n_kv) to_fp16 pass goodbadwolf's
// comment in the same issue points at).  The API is indices-in: no mask is
// built or re-scanned.
//
// Grid (split, KV head, token).  A CTA owns up to kCS consecutive entries of
// the token's cell list: it gathers their K and V rows for its KV head with
// 16-byte cp.async copies (all copies in flight at once), computes the 8
// query heads' scores, a local softmax (max m, sum l) and the unnormalised
// P.V, and writes the partial (m, l, o[256]) per head.  k_combine merges the
// partials of a token with log-sum-exp weights.  fp32 accumulation.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kAttnThreads = 256;
constexpr int kCS = 64;   // cells per split

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <bool kQ8>
struct AttnSmem;

template <>
struct AttnSmem<false> {
  __half k[kCS][kHeadDim];
  __half v[kCS][kHeadDim];
  float q[kGqa][kHeadDim];
  float p[kCS][kGqa];
  int cell[kCS];
  float m[kGqa], l[kGqa];
};

template <>
struct AttnSmem<true> {
  int8_t k[kCS][kHeadDim];
  int8_t v[kCS][kHeadDim];
  __half ks[kCS][kHeadDim / 32];
  __half vs[kCS][kHeadDim / 32];
  float q[kGqa][kHeadDim];
  float p[kCS][kGqa];
  int cell[kCS];
  float m[kGqa], l[kGqa];
};

__device__ __forceinline__ void h8_to_f(uint4 raw, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

__device__ __forceinline__ void q8_to_f(uint2 raw, float scale, float* f) {
  const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = scale * (float)b[i];
}

template <bool kQ8>
__global__ void __launch_bounds__(kAttnThreads)
k_attn_split(const AttnArgs a, float* __restrict__ part_o, float2* __restrict__ part_ml,
             int ns_max, unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem<kQ8>& sm = *reinterpret_cast<AttnSmem<kQ8>*>(smem_raw);

  const int s = blockIdx.x, g = blockIdx.y, t = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.n_kv_heads, Hq = G * kGqa;
  int cnt = a.count[t];
  cnt = cnt < 0 ? 0 : (cnt > a.cells_pitch ? a.cells_pitch : cnt);
  const int c0 = s * kCS;
  if (c0 >= cnt) return;
  const int nv = min(kCS, cnt - c0);

  if (tid < kCS) {
    int c = -1;
    if (tid < nv) {
      c = a.cells[(int64_t)t * a.cells_pitch + c0 + tid];
      if (c < 0 || c >= a.n_cells) {
        atomicOr(err, kErrCell);
        c = -1;
      }
    }
    sm.cell[tid] = c;
  }
  {
    const __half2* qg = reinterpret_cast<const __half2*>(a.q + ((int64_t)t * Hq + g * kGqa) * kHeadDim);
    float* qs = &sm.q[0][0];
    for (int i = tid; i < kGqa * kHeadDim / 2; i += kAttnThreads) {
      const float2 f = __half22float2(qg[i]);
      qs[2 * i] = f.x;
      qs[2 * i + 1] = f.y;
    }
  }
  __syncthreads();

  // Gather: K first (own commit group) so QK can start while V is in flight.
  if constexpr (!kQ8) {
    const __half* kb = static_cast<const __half*>(a.k_cache);
    const __half* vb = static_cast<const __half*>(a.v_cache);
    for (int id = tid; id < kCS * 32; id += kAttnThreads) {
      const int row = id >> 5, col = id & 31, c = sm.cell[row];
      cp_async16(&sm.k[row][col * 8], kb + ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + col * 8, c >= 0);
    }
    cp_async_commit();
    for (int id = tid; id < kCS * 32; id += kAttnThreads) {
      const int row = id >> 5, col = id & 31, c = sm.cell[row];
      cp_async16(&sm.v[row][col * 8], vb + ((int64_t)(c < 0 ? 0 : c) * G + g) * kHeadDim + col * 8, c >= 0);
    }
    cp_async_commit();
  } else {
    const int8_t* kq = static_cast<const int8_t*>(a.k_cache);
    const int8_t* vq = static_cast<const int8_t*>(a.v_cache);
    const int64_t nq = a.n_cells * (int64_t)G * kHeadDim;
    const __half* kd = reinterpret_cast<const __half*>(kq + nq);
    const __half* vd = reinterpret_cast<const __half*>(vq + nq);
    for (int id = tid; id < kCS * 17; id += kAttnThreads) {
      const int row = id / 17, col = id % 17, c = sm.cell[row];
      const int64_t cg = (int64_t)(c < 0 ? 0 : c) * G + g;
      if (col < 16) cp_async16(&sm.k[row][col * 16], kq + cg * kHeadDim + col * 16, c >= 0);
      else cp_async16(&sm.ks[row][0], kd + cg * (kHeadDim / 32), c >= 0);
    }
    cp_async_commit();
    for (int id = tid; id < kCS * 17; id += kAttnThreads) {
      const int row = id / 17, col = id % 17, c = sm.cell[row];
      const int64_t cg = (int64_t)(c < 0 ? 0 : c) * G + g;
      if (col < 16) cp_async16(&sm.v[row][col * 16], vq + cg * kHeadDim + col * 16, c >= 0);
      else cp_async16(&sm.vs[row][0], vd + cg * (kHeadDim / 32), c >= 0);
    }
    cp_async_commit();
  }
  cp_async_wait<1>();
  __syncthreads();

  // Scores: warp w owns cells 8w..8w+7, lane l owns dims 8l..8l+7.
  {
    float qr[kGqa][8];
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const float4 x = *reinterpret_cast<const float4*>(&sm.q[h][8 * lane]);
      const float4 y = *reinterpret_cast<const float4*>(&sm.q[h][8 * lane + 4]);
      qr[h][0] = x.x; qr[h][1] = x.y; qr[h][2] = x.z; qr[h][3] = x.w;
      qr[h][4] = y.x; qr[h][5] = y.y; qr[h][6] = y.z; qr[h][7] = y.w;
    }
    float v[64];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int cell = warp * 8 + cc;
      float kf[8];
      if constexpr (!kQ8) {
        h8_to_f(*reinterpret_cast<const uint4*>(&sm.k[cell][8 * lane]), kf);
      } else {
        q8_to_f(*reinterpret_cast<const uint2*>(&sm.k[cell][8 * lane]),
                __half2float(sm.ks[cell][lane >> 2]), kf);
      }
#pragma unroll
      for (int h = 0; h < kGqa; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) acc = fmaf(qr[h][d], kf[d], acc);
        v[cc * 8 + h] = acc;
      }
    }
    // Reduce-scatter the 64 (cell, head) partial dots over the 32 lanes:
    // lane L ends with entries 2L and 2L+1, i.e. cell L/4, heads 2(L%4)+{0,1}.
#pragma unroll
    for (int m = 16, n = 32; m >= 1; m >>= 1, n >>= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float send = upper ? v[i] : v[i + n];
        const float keep = upper ? v[i + n] : v[i];
        v[i] = keep + __shfl_xor_sync(kFull, send, m);
      }
    }
    const int cell = warp * 8 + (lane >> 2);
    const int h0 = 2 * (lane & 3);
    const bool valid = sm.cell[cell] >= 0;
    sm.p[cell][h0] = valid ? v[0] * a.attn_scale : -INFINITY;
    sm.p[cell][h0 + 1] = valid ? v[1] * a.attn_scale : -INFINITY;
  }
  __syncthreads();

  // Local softmax: warp h handles head h over the kCS cells.
  {
    const int h = warp;
    const float x0 = sm.p[lane][h], x1 = sm.p[lane + 32][h];
    float m = fmaxf(x0, x1);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    const float e0 = (m == -INFINITY) ? 0.f : expf(x0 - m);
    const float e1 = (m == -INFINITY) ? 0.f : expf(x1 - m);
    float l = e0 + e1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
    sm.p[lane][h] = e0;
    sm.p[lane + 32][h] = e1;
    if (lane == 0) {
      sm.m[h] = m;
      sm.l[h] = l;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // P.V: thread d owns output dim d for the 8 heads.
  {
    const int d = tid;
    float o[kGqa];
#pragma unroll
    for (int h = 0; h < kGqa; ++h) o[h] = 0.f;
    for (int c = 0; c < nv; ++c) {
      float vv;
      if constexpr (!kQ8) vv = __half2float(sm.v[c][d]);
      else vv = __half2float(sm.vs[c][d >> 5]) * (float)sm.v[c][d];
      const float4 p0 = *reinterpret_cast<const float4*>(&sm.p[c][0]);
      const float4 p1 = *reinterpret_cast<const float4*>(&sm.p[c][4]);
      o[0] = fmaf(p0.x, vv, o[0]); o[1] = fmaf(p0.y, vv, o[1]);
      o[2] = fmaf(p0.z, vv, o[2]); o[3] = fmaf(p0.w, vv, o[3]);
      o[4] = fmaf(p1.x, vv, o[4]); o[5] = fmaf(p1.y, vv, o[5]);
      o[6] = fmaf(p1.z, vv, o[6]); o[7] = fmaf(p1.w, vv, o[7]);
    }
#pragma unroll
    for (int h = 0; h < kGqa; ++h) {
      const int64_t row = ((int64_t)t * Hq + g * kGqa + h) * ns_max + s;
      part_o[row * kHeadDim + d] = o[h];
    }
    if (tid < kGqa) {
      const int64_t row = ((int64_t)t * Hq + g * kGqa + tid) * ns_max + s;
      part_ml[row] = make_float2(sm.m[tid], sm.l[tid]);
    }
  }
}

__global__ void __launch_bounds__(kHeadDim)
k_combine(const AttnArgs a, const float* __restrict__ part_o, const float2* __restrict__ part_ml, int ns_max) {
  const int h = blockIdx.x, t = blockIdx.y, d = threadIdx.x;
  const int Hq = a.n_kv_heads * kGqa;
  int cnt = a.count[t];
  cnt = cnt < 0 ? 0 : (cnt > a.cells_pitch ? a.cells_pitch : cnt);
  const int ns = (int)ceil_div(cnt, kCS);
  const int64_t row0 = ((int64_t)t * Hq + h) * ns_max;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, part_ml[row0 + s].x);
  float L = 0.f, o = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const float2 ml = part_ml[row0 + s];
      const float w = (ml.x == -INFINITY) ? 0.f : expf(ml.x - M);
      L = fmaf(w, ml.y, L);
      o = fmaf(w, part_o[(row0 + s) * kHeadDim + d], o);
    }
  }
  a.out[((int64_t)t * Hq + h) * kHeadDim + d] = L > 0.f ? o / L : 0.f;
}

template <bool kQ8>
cudaError_t launch_split(const AttnArgs& a, float* po, float2* pml, int ns_max, unsigned* err,
                         cudaStream_t stream) {
  const size_t smem = sizeof(AttnSmem<kQ8>);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_split<kQ8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 grid((unsigned)ns_max, (unsigned)a.n_kv_heads, (unsigned)a.n_tokens);
  prof_before(kKAttn, stream);
  k_attn_split<kQ8><<<grid, kAttnThreads, smem, stream>>>(a, po, pml, ns_max, err);
  prof_after(kKAttn, stream);
  return cudaGetLastError();
}

}  // namespace

size_t attn_workspace_bytes(int n_tokens, int n_q_heads, int cells_pitch) {
  const int64_t ns = ceil_div(cells_pitch, kCS);
  const int64_t rows = (int64_t)n_tokens * n_q_heads * ns;
  return (size_t)round_up(rows * kHeadDim * (int64_t)sizeof(float), 256) +
         (size_t)round_up(rows * (int64_t)sizeof(float2), 256);
}

cudaError_t launch_sparse_attn(const AttnArgs& a, void* ws, unsigned* err, cudaStream_t stream) {
  if (a.n_tokens <= 0) return cudaSuccess;
  const int ns_max = (int)ceil_div(a.cells_pitch, kCS);
  const int Hq = a.n_kv_heads * kGqa;
  const int64_t rows = (int64_t)a.n_tokens * Hq * ns_max;
  float* po = static_cast<float*>(ws);
  float2* pml = reinterpret_cast<float2*>(static_cast<char*>(ws) +
                                          round_up(rows * kHeadDim * (int64_t)sizeof(float), 256));
  cudaError_t e = a.kv_q8 ? launch_split<true>(a, po, pml, ns_max, err, stream)
                          : launch_split<false>(a, po, pml, ns_max, err, stream);
  if (e != cudaSuccess) return e;
  prof_before(kKCombine, stream);
  k_combine<<<dim3((unsigned)Hq, (unsigned)a.n_tokens), kHeadDim, 0, stream>>>(a, po, pml, ns_max);
  prof_after(kKCombine, stream);
  return cudaGetLastError();
}

}  // namespace qsa
