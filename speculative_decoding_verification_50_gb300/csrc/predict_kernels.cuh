// a4 outcome prediction and a5 hit check ("Speculative Speculative Decoding"
// §4.1.1 Saguaro verification-outcome prediction; §3.1 cache hit).
//
// A unit is one draft row (b, k), k in [0, K], owned by a cluster of C CTAs,
// each streaming a vocabulary slice once.  Every warp keeps a sorted top-F
// list distributed over its lanes (lane f holds entry f); a lane's logit
// enters the list only if it reaches the list's current F-th entry (one
// compare and a ballot per element in the common case).  Lists are merged
// warp -> CTA (shared memory) -> cluster (distributed shared memory, rank 0).
// The order is (logit descending, index ascending), so the result is the
// unique top-F set regardless of the order candidates arrive in.
#pragma once

#include <climits>

#include "specv_common.cuh"

namespace specv {

struct PredictParams {
  const void* zd;
  int64_t d_bs, d_rs;
  const int32_t* tokens;
  int32_t* keys;
  float* key_logits;
  int32_t* unit_status;  // [B*(K+1)] or null
  int32_t B, K, V, F, C, L;
};

__device__ __forceinline__ bool key_beats(float av, int32_t ai, float bv, int32_t bi) {
  return av > bv || (av == bv && ai < bi);
}

// Sorted list over a warp; empty entries are (-inf, INT_MAX), below any key.
struct WarpTopF {
  float v;
  int32_t i;
  float tv;  // entry F-1 (the admission threshold), same in every lane
  int32_t ti;
  __device__ __forceinline__ void init() {
    v = neg_inf();
    i = INT_MAX;
    tv = neg_inf();
    ti = INT_MAX;
  }
  // Insert candidate (cv, ci), warp-uniform arguments.
  __device__ __forceinline__ void insert(float cv, int32_t ci, int F, int lane) {
    const bool ahead = lane < F && key_beats(v, i, cv, ci);
    const int pos = __popc(__ballot_sync(0xffffffffu, ahead));
    if (pos >= F) return;
    const float uv = __shfl_up_sync(0xffffffffu, v, 1);
    const int32_t ui = __shfl_up_sync(0xffffffffu, i, 1);
    if (lane > pos && lane < F) {
      v = uv;
      i = ui;
    } else if (lane == pos) {
      v = cv;
      i = ci;
    }
    tv = __shfl_sync(0xffffffffu, v, F - 1);
    ti = __shfl_sync(0xffffffffu, i, F - 1);
  }
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) predict_units_kernel(const PredictParams P) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  constexpr int U = 2;
  __shared__ float wv[kWarps][32];
  __shared__ int32_t wi[kWarps][32];
  __shared__ float cv[32];
  __shared__ int32_t ci[32];
  __shared__ int32_t cbad;
  __shared__ int32_t wbad[kWarps];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = P.C;
  const int64_t u = blockIdx.x / C;
  const int K = P.K, F = P.F;
  const int b = static_cast<int>(u / (K + 1));
  const int k = static_cast<int>(u % (K + 1));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int excl = (k < K) ? P.tokens[static_cast<int64_t>(b) * K + k] : -1;
  const bool bad_token = (k < K) && (excl < 0 || excl >= P.V);

  const void* row = static_cast<const char*>(P.zd) +
                    (static_cast<int64_t>(b) * P.d_bs + static_cast<int64_t>(k) * P.d_rs) * E::ES;
  const int64_t v0 = static_cast<int64_t>(rank) * P.L;
  const int64_t v1 = min(static_cast<int64_t>(P.V), v0 + P.L);
  const int nv = v1 > v0 ? static_cast<int>((v1 - v0 + VW - 1) / VW) : 0;
  const int ntl = (nv + kThreads - 1) / kThreads;

  WarpTopF L;
  L.init();
  int bad = 0;
  if (!bad_token) {
    for (int t0 = 0; t0 < ntl; t0 += U) {
      typename E::Vec w[U];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const int j = (t0 + uu) * kThreads + threadIdx.x;
        if (j < nv) w[uu] = load_vec<DT, VEC>(row, v0, v1, j);
      }
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        if (t0 + uu >= ntl) break;  // uniform
        const int j = (t0 + uu) * kThreads + threadIdx.x;
        float z[VW];
        if (j < nv) {
          E::unpack(w[uu], z);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) z[e] = neg_inf();
        }
        const int32_t base = static_cast<int32_t>(v0) + j * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const int32_t vi = base + e;
          const bool valid = j < nv && vi < v1;
          bad |= valid && !(z[e] < pos_inf());
          const bool pass = valid && z[e] >= L.tv && vi != excl;
          unsigned m = __ballot_sync(0xffffffffu, pass);
          while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float zz = __shfl_sync(0xffffffffu, z[e], src);
            const int32_t ii = __shfl_sync(0xffffffffu, vi, src);
            L.insert(zz, ii, F, lane);
          }
        }
      }
    }
  }
  // warp lists -> shared memory; warp 0 merges them into the CTA list
  wv[warp][lane] = L.v;
  wi[warp][lane] = L.i;
  bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) wbad[warp] = bad;
  __syncthreads();
  if (warp == 0) {
    WarpTopF M;
    M.v = wv[0][lane];
    M.i = wi[0][lane];
    M.tv = __shfl_sync(0xffffffffu, M.v, F - 1);
    M.ti = __shfl_sync(0xffffffffu, M.i, F - 1);
    for (int w = 1; w < kWarps; ++w)
      for (int f = 0; f < F; ++f) {
        const float zz = wv[w][f];
        const int32_t ii = wi[w][f];
        if (key_beats(zz, ii, M.tv, M.ti)) M.insert(zz, ii, F, lane);
      }
    cv[lane] = M.v;
    ci[lane] = M.i;
    if (lane == 0) {
      int bb = 0;
      for (int w = 0; w < kWarps; ++w) bb |= wbad[w];
      cbad = bb;
    }
  }
  cluster.sync();  // (1) CTA lists visible cluster-wide
  if (rank == 0 && warp == 0) {
    WarpTopF M;
    M.v = cv[lane];
    M.i = ci[lane];
    M.tv = __shfl_sync(0xffffffffu, M.v, F - 1);
    M.ti = __shfl_sync(0xffffffffu, M.i, F - 1);
    int bb = cbad;
    for (int r = 1; r < C; ++r) {
      const float* rv = cluster.map_shared_rank(cv, r);
      const int32_t* ri = cluster.map_shared_rank(ci, r);
      bb |= *cluster.map_shared_rank(&cbad, r);
      for (int f = 0; f < F; ++f) {
        const float zz = rv[f];
        const int32_t ii = ri[f];
        if (key_beats(zz, ii, M.tv, M.ti)) M.insert(zz, ii, F, lane);
      }
    }
    const int status = (bad_token ? kBadToken : 0) | (bb ? kNonFinite : 0);
    if (lane < F) {
      const int64_t o = u * F + lane;
      const bool ok = status == 0 && M.i != INT_MAX;
      P.keys[o] = ok ? M.i : -1;
      if (P.key_logits) P.key_logits[o] = ok ? M.v : neg_inf();
    }
    if (lane == 0 && P.unit_status) P.unit_status[u] = status;
  }
  cluster.sync();  // (2) no CTA exits while rank 0 reads its list
}

__global__ void predict_finalize_kernel(const int32_t* __restrict__ unit_status, int B, int K,
                                        int32_t* __restrict__ row_status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int s = 0;
  for (int k = 0; k <= K; ++k) s |= unit_status[static_cast<int64_t>(b) * (K + 1) + k];
  row_status[b] = s;
}

__global__ void check_hit_kernel(int B, int K, int F, const int32_t* __restrict__ keys,
                                 const int32_t* __restrict__ accept_len,
                                 const int32_t* __restrict__ out_tokens,
                                 uint8_t* __restrict__ hit) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = accept_len[b];
  uint8_t h = 0;
  if (n >= 0 && n <= K) {
    const int t = out_tokens[static_cast<int64_t>(b) * (K + 1) + n];
    if (t >= 0) {
      const int32_t* kk = keys + (static_cast<int64_t>(b) * (K + 1) + n) * F;
      for (int f = 0; f < F; ++f) h |= (kk[f] == t);
    }
  }
  hit[b] = h;
}

}  // namespace specv
