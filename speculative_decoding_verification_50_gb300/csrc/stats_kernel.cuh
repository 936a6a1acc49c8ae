// Kernel A of the hot path: one streaming pass over every logit row.
//
// a1 row statistics ("Lecture 5 - Speculative Decoding and SpecInfer" §2.1:
// temperature T gives softmax(z/T), greedy gives the one-hot argmax) and, in
// the modes that predict outcomes, the per-chunk candidates for a4 ("Speculative
// Speculative Decoding" §4.1.1: top-F draft tokens at each lookahead, the token
// sent for verification there excluded).
//
// A unit is one (batch row b, position i), i in [0, K]; a CTA owns one chunk of
// the unit's rows (target row i and/or draft row i): `iters` trips of kVecs
// 16-byte vectors per row per thread.  The loop is software-pipelined: the next
// trip's loads are in flight while the current trip is consumed, so a thread
// keeps 2*kVecs vectors per row outstanding; there is no shared staging and no
// cluster, so CTAs are small and many.
//
// Per chunk the CTA writes a ChunkRec: online (max, sum 2^((z-max) log2(e)/T))
// of each row, or its first argmax for greedy rows.  With outcome prediction it
// also writes the chunk's own top-F of the draft row: the (F+1)-th largest of a
// warp's per-thread maxima bounds the chunk's top-F from below, so only the few
// threads whose maximum reaches the bound read their logits again (from L2,
// just streamed) and push the qualifying ones into shared memory, where they
// are ranked in parallel.
#pragma once

#include "specv_device.cuh"

namespace specv {

enum : int { kModeVerify = 0, kModeSsd = 1, kModePredict = 2 };
constexpr int kVecs = 2;  // 16-byte vectors per row per thread per loop trip

struct ChunkRec {        // 48 bytes per (unit, chunk)
  float mt, st, md, sd;  // temperature rows: max and sum of 2^((z-max)c)
  float bt, bd;          // greedy rows: best logit
  int32_t it, id;        // greedy rows: first index of the best logit
  int32_t bad;           // bit 0: NaN or +inf seen in a greedy row (T > 0: shows
                         // as a NaN sum); bit 1: a staged copy did not land in time
  int32_t pad[3];
};
static_assert(sizeof(ChunkRec) == 48, "ChunkRec layout");

struct StatsParams {
  const void* zt;
  int64_t t_bs, t_rs;
  const void* zd;
  int64_t d_bs, d_rs;
  const int32_t* tokens;
  const float* temp;
  ChunkRec* recs;     // [units * nchunk]
  float* cand_v;      // [units * nchunk * F] (predict / ssd)
  int32_t* cand_i;
  int32_t B, K, V, F, nchunk, chunk, iters;  // chunk = iters * kVecs * 256 * VW logits
};

// log2(e)/T for a valid temperature; greedy rows and bad temperatures use 1.
__device__ __forceinline__ float temp_scale(float T) {
  return (T > 0.f && T < pos_inf()) ? __fdiv_rn(1.44269504088896341f, T) : 1.f;
}

template <int DT, bool VEC>
__device__ __forceinline__ void load_trip(const void* row, int64_t v0, int64_t v1, int nv, int it,
                                          typename Elem<DT>::Vec (&w)[kVecs]) {
#pragma unroll
  for (int k = 0; k < kVecs; ++k) {
    const int j = (it * kVecs + k) * kThreads + threadIdx.x;
    if (j < nv) w[k] = load_vec<DT, VEC>(row, v0, v1, j);
  }
}

template <int DT, bool GREEDY>
__device__ __forceinline__ void consume_trip(const typename Elem<DT>::Vec (&w)[kVecs], int nv,
                                             int it, int64_t v0, float c,
                                             Soft<Elem<DT>::VW>& s, Arg& a) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
#pragma unroll
  for (int k = 0; k < kVecs; ++k) {
    const int j = (it * kVecs + k) * kThreads + threadIdx.x;
    if (j < nv) {
      float z[VW];
      E::unpack(w[k], z);
      if (GREEDY) a.add(z, static_cast<int32_t>(v0) + j * VW); else s.add(z, c);
    }
  }
}

// Streams the CTA's chunk of one or two rows (software-pipelined).
template <int DT, bool VEC, bool GREEDY, bool KT>
__device__ __forceinline__ void stream_chunk(const void* rowt, const void* rowd, bool has_d,
                                             int64_t v0, int64_t v1, int nv, int iters, float c,
                                             Soft<Elem<DT>::VW>& st, Soft<Elem<DT>::VW>& sd,
                                             Arg& at, Arg& ad) {
  using Vec = typename Elem<DT>::Vec;
  Vec at0[kVecs], ad0[kVecs], at1[kVecs], ad1[kVecs];
  if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, 0, at0);
  if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, 0, ad0);
  for (int it = 0; it < iters; it += 2) {
    if (it + 1 < iters) {
      if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, it + 1, at1);
      if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, it + 1, ad1);
    }
    if (KT) consume_trip<DT, GREEDY>(at0, nv, it, v0, c, st, at);
    if (has_d) consume_trip<DT, GREEDY>(ad0, nv, it, v0, c, sd, ad);
    if (it + 1 < iters) {
      if (it + 2 < iters) {
        if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, it + 2, at0);
        if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, it + 2, ad0);
      }
      if (KT) consume_trip<DT, GREEDY>(at1, nv, it + 1, v0, c, st, at);
      if (has_d) consume_trip<DT, GREEDY>(ad1, nv, it + 1, v0, c, sd, ad);
    }
  }
}

// ---- TMA ring (16-byte aligned rows) ----------------------------------------
// A trip is kVecs*256 16-byte vectors of each row; stage s of the ring holds
// one trip of every streamed row.  Thread 0 keeps up to kStages trips in
// flight as 1-D bulk copies completing on the stage's mbarrier; all threads
// consume a stage from shared memory, meet at a CTA barrier, and thread 0
// refills the stage with the trip kStages ahead.  The vector -> thread mapping
// is that of the register path, so results are identical.
constexpr int kStages = 4;
constexpr int kTripBytes = kVecs * kThreads * 16;  // per row per trip (8 KB)

struct Ring {
  uint64_t full[kStages];
};

// Issue trip t of the chunk into stage t % kStages.  Bytes past the last whole
// 16-byte unit of the chunk are left to the consumers (plain loads).
__device__ __forceinline__ void ring_issue(Ring& R, unsigned char* stages, int t,
                                          const char* rowt, const char* rowd, int64_t first,
                                          int64_t n_bytes_chunk) {
  const int st = t % kStages;
  const int64_t off = static_cast<int64_t>(t) * kTripBytes;
  int64_t bytes = n_bytes_chunk - off;
  if (bytes > kTripBytes) bytes = kTripBytes;
  bytes &= ~static_cast<int64_t>(15);
  if (bytes < 0) bytes = 0;
  const uint32_t b32 = static_cast<uint32_t>(bytes);
  mbar_arrive_expect_tx(&R.full[st], b32 * ((rowt ? 1u : 0u) + (rowd ? 1u : 0u)));
  if (b32) {
    unsigned char* base = stages + static_cast<int64_t>(st) * 2 * kTripBytes;
    if (rowt) bulk_load(base, rowt + first + off, b32, &R.full[st]);
    if (rowd) bulk_load(base + kTripBytes, rowd + first + off, b32, &R.full[st]);
  }
}

// Vector k of this thread in stage buffer `buf` for trip t: from shared
// memory, or element by element from global memory for the ragged tail that
// no bulk copy covered; -inf beyond the chunk.
template <int DT>
__device__ __forceinline__ typename Elem<DT>::Vec ring_vec(const unsigned char* buf, const char* row,
                                                           int64_t v0, int64_t v1, int t, int k,
                                                           int64_t covered_elems) {
  using E = Elem<DT>;
  const int jl = k * kThreads + threadIdx.x;               // vector within the trip
  const int64_t e = v0 + (static_cast<int64_t>(t) * kVecs * kThreads + jl) * E::VW;  // first element
  if (e + E::VW <= v0 + covered_elems) return reinterpret_cast<const typename E::Vec*>(buf)[jl];
  return E::gather(row, e, v1);
}

template <int DT, bool GREEDY, bool KT>
__device__ __forceinline__ bool stream_chunk_tma(Ring& R, unsigned char* stages, const char* rowt,
                                                 const char* rowd, bool has_d, int64_t v0,
                                                 int64_t v1, int nv, float c,
                                                 Soft<Elem<DT>::VW>& st, Soft<Elem<DT>::VW>& sd,
                                                 Arg& at, Arg& ad) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  const int ntr = (nv + kVecs * kThreads - 1) / (kVecs * kThreads);
  const int64_t first = v0 * E::ES;
  const int64_t n_bytes = (v1 - v0) * E::ES;
  const int64_t covered = (n_bytes & ~static_cast<int64_t>(15)) / E::ES;  // elements in bulk copies
  const char* rt = KT ? rowt : nullptr;
  const char* rd = has_d ? rowd : nullptr;
  if (threadIdx.x == 0) {
    for (int s2 = 0; s2 < kStages; ++s2) mbar_init(&R.full[s2], 1);
    fence_mbar_init();
    for (int t = 0; t < ntr && t < kStages; ++t) ring_issue(R, stages, t, rt, rd, first, n_bytes);
  }
  __syncthreads();
  bool ok = true;
  for (int t = 0; t < ntr; ++t) {
    const int s2 = t % kStages;
    if (!mbar_wait_bounded(&R.full[s2], static_cast<uint32_t>((t / kStages) & 1))) ok = false;
    const unsigned char* base = stages + static_cast<int64_t>(s2) * 2 * kTripBytes;
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const int j = (t * kVecs + k) * kThreads + threadIdx.x;
      if (j < nv) {
        float z[VW];
        const int32_t b0 = static_cast<int32_t>(v0) + j * VW;
        if (KT) {
          E::unpack(ring_vec<DT>(base, rowt, v0, v1, t, k, covered), z);
          if (GREEDY) at.add(z, b0); else st.add(z, c);
        }
        if (has_d) {
          E::unpack(ring_vec<DT>(base + kTripBytes, rowd, v0, v1, t, k, covered), z);
          if (GREEDY) ad.add(z, b0); else sd.add(z, c);
        }
      }
    }
    // Stage s2 consumed by every thread.  If any wait gave up, issue nothing
    // more, give the copies in flight a bounded wait to land, and report.
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0)
        for (int t2 = t; t2 < ntr && t2 < t + kStages; ++t2)
          mbar_wait_bounded(&R.full[t2 % kStages], static_cast<uint32_t>((t2 / kStages) & 1));
      __syncthreads();
      return false;
    }
    if (threadIdx.x == 0 && t + kStages < ntr) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue(R, stages, t + kStages, rt, rd, first, n_bytes);
    }
  }
  return ok;
}

template <int DT, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads, DT == 0 ? 3 : 4) stats_kernel(const StatsParams P) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  constexpr bool kT = MODE != kModePredict;
  constexpr bool kTopF = MODE != kModeVerify;
  __shared__ ChunkRec wrec[kWarps];
  __shared__ float wthr[kWarps];
  __shared__ float wl_v[kWarps][kMaxF];
  __shared__ int32_t wl_i[kWarps][kMaxF];
  __shared__ KeyScratch KS;

  const int64_t u = blockIdx.x / P.nchunk;
  const int ch = static_cast<int>(blockIdx.x % P.nchunk);
  const int K = P.K;
  const int b = static_cast<int>(u / (K + 1));
  const int i = static_cast<int>(u % (K + 1));
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool has_d = (MODE == kModeVerify) ? (i < K) : true;
  const float T = kT ? P.temp[b] : 0.f;
  const bool greedy = !kT || T == 0.f;
  const float c = greedy ? 1.f : temp_scale(T);

  const char* rowt = kT ? static_cast<const char*>(P.zt) +
                              (static_cast<int64_t>(b) * P.t_bs + static_cast<int64_t>(i) * P.t_rs) * E::ES
                        : nullptr;
  const char* rowd = has_d ? static_cast<const char*>(P.zd) +
                                 (static_cast<int64_t>(b) * P.d_bs + static_cast<int64_t>(i) * P.d_rs) * E::ES
                           : nullptr;
  const int64_t v0 = static_cast<int64_t>(ch) * P.chunk;
  const int64_t v1 = min(static_cast<int64_t>(P.V), v0 + P.chunk);
  const int nv = static_cast<int>((v1 - v0 + VW - 1) / VW);

  const int excl = (kTopF && i < K) ? P.tokens[static_cast<int64_t>(b) * K + i] : -1;
  Soft<VW> st, sd;
  Arg at, ad;
  st.init();
  sd.init();
  at.init();
  ad.init();
  int copy_bad = 0;  // bit 1: a staged copy did not land in time
  if (VEC) {
    extern __shared__ __align__(128) unsigned char stages[];
    __shared__ Ring ring;
    const bool ok = greedy
        ? stream_chunk_tma<DT, true, kT>(ring, stages, rowt, rowd, has_d, v0, v1, nv, c, st, sd, at, ad)
        : stream_chunk_tma<DT, false, kT>(ring, stages, rowt, rowd, has_d, v0, v1, nv, c, st, sd, at, ad);
    copy_bad = ok ? 0 : 2;  // every thread of the CTA returns the same verdict
  } else if (greedy) {
    stream_chunk<DT, VEC, true, kT>(rowt, rowd, has_d, v0, v1, nv, P.iters, c, st, sd, at, ad);
  } else {
    stream_chunk<DT, VEC, false, kT>(rowt, rowd, has_d, v0, v1, nv, P.iters, c, st, sd, at, ad);
  }

  // ---- reduce: warp, then CTA (warp 0 over the eight warp partials) --------
  const float tmax_d = greedy ? ad.best : sd.m;  // this thread's draft maximum
  if (greedy) {
    float bt = at.best, bd = ad.best;
    int32_t it = at.idx, id = ad.idx;
    warp_arg_all(bt, it);
    warp_arg_all(bd, id);
    const int bad = __any_sync(0xffffffffu, at.bad | ad.bad);
    if (lane == 0) {
      wrec[warp].bt = bt; wrec[warp].it = it; wrec[warp].bd = bd; wrec[warp].id = id;
      wrec[warp].bad = bad;
    }
  } else {
    float mt = st.m, s_t = st.total(), md = sd.m, s_d = sd.total();
    warp_soft_all(mt, s_t, c);
    warp_soft_all(md, s_d, c);
    if (lane == 0) {
      wrec[warp].mt = mt; wrec[warp].st = s_t; wrec[warp].md = md; wrec[warp].sd = s_d;
    }
  }
  if (kTopF) {
    if (threadIdx.x == 0) KS.count = 0;
    if (threadIdx.x < P.F) {
      KS.out_v[threadIdx.x] = neg_inf();
      KS.out_i[threadIdx.x] = INT_MAX;
    }
    // (F+1)-th largest per-thread max of this warp: a lower bound on the
    // chunk's (F+1)-th largest draft logit, hence on its top-F without x.
    float s = tmax_d;
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
      for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, s, j2);
        const bool take_max = ((lane & k2) == 0) == ((lane & j2) == 0);
        s = take_max ? fmaxf(s, o) : fminf(s, o);
      }
    }
    const float tw = (P.F < 32) ? __shfl_sync(0xffffffffu, s, P.F) : neg_inf();
    if (lane == 0) wthr[warp] = tw;
  }
  __syncthreads();
  if (warp == 0) {
    ChunkRec r;
    r.mt = kNegMax; r.st = 0.f; r.md = kNegMax; r.sd = 0.f;
    r.bt = neg_inf(); r.it = INT_MAX; r.bd = neg_inf(); r.id = INT_MAX; r.bad = 0;
    r.pad[0] = r.pad[1] = r.pad[2] = 0;
    if (greedy) {
      float bt = neg_inf(), bd = neg_inf();
      int32_t it = INT_MAX, id = INT_MAX;
      int bad = 0;
      if (lane < kWarps) {
        bt = wrec[lane].bt; it = wrec[lane].it; bd = wrec[lane].bd; id = wrec[lane].id;
        bad = wrec[lane].bad;
      }
      warp_arg_all(bt, it);
      warp_arg_all(bd, id);
      r.bt = bt; r.it = it; r.bd = bd; r.id = id;
      r.bad = __any_sync(0xffffffffu, bad);
    } else {
      float mt = kNegMax, s_t = 0.f, md = kNegMax, s_d = 0.f;
      if (lane < kWarps) {
        mt = wrec[lane].mt; s_t = wrec[lane].st; md = wrec[lane].md; s_d = wrec[lane].sd;
      }
      warp_soft_all(mt, s_t, c);
      warp_soft_all(md, s_d, c);
      r.mt = mt; r.st = s_t; r.md = md; r.sd = s_d;
    }
    r.bad |= copy_bad;
    if (lane == 0) P.recs[blockIdx.x] = r;
  }

  if (kTopF) {
    // Only threads whose maximum reaches the bound can hold a top-F logit.
    // Their logits are read again (from L2, just streamed) by their whole
    // warp -- lane k fetches the candidate thread's k-th vector -- and the
    // qualifying ones are pushed into a shared buffer, ranked in parallel.
    // Too many qualifiers (ties at the bound), or no finite bound at all
    // (F = 32, masked rows), take the exact warp-list path.
    const int F = P.F;
    float thr = wthr[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) thr = fmaxf(thr, wthr[w]);
    const bool bounded = thr > kNegMax;
    const int ntrips = P.iters * kVecs;
    unsigned cm = __ballot_sync(0xffffffffu, bounded && tmax_d >= thr);
    while (cm) {
      const int owner = warp * 32 + __ffs(cm) - 1;
      cm &= cm - 1;
      for (int k = lane; k < ntrips; k += 32) {
        const int j = k * kThreads + owner;
        if (j < nv) {
          float z[VW];
          E::unpack(load_vec<DT, VEC>(rowd, v0, v1, j), z);
          const int32_t base = static_cast<int32_t>(v0) + j * VW;
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const int32_t vi = base + e;
            if (vi < v1 && vi != excl && z[e] >= thr) {
              const int slot = atomicAdd(&KS.count, 1);
              if (slot < kCandCap) {
                KS.v[slot] = z[e];
                KS.i[slot] = vi;
              }
            }
          }
        }
      }
    }
    if (!bounded && threadIdx.x == 0) KS.count = kCandCap + 1;  // exact path below
    __syncthreads();
    const int m = KS.count;
    float* outv = P.cand_v + static_cast<int64_t>(blockIdx.x) * F;
    int32_t* outi = P.cand_i + static_cast<int64_t>(blockIdx.x) * F;
    if (m <= kCandCap) {
      for (int e = threadIdx.x; e < m; e += kThreads) {
        const float v = KS.v[e];
        const int32_t ii = KS.i[e];
        int rank = 0;
        for (int o = 0; o < m; ++o) rank += key_beats(KS.v[o], KS.i[o], v, ii);
        if (rank < F) {
          KS.out_v[rank] = v;
          KS.out_i[rank] = ii;
        }
      }
      __syncthreads();
      if (threadIdx.x < F) {
        outv[threadIdx.x] = KS.out_v[threadIdx.x];
        outi[threadIdx.x] = KS.out_i[threadIdx.x];
      }
    } else {
      WarpTopF L;
      L.init();
      for (int k = 0; k < ntrips; ++k) {
        const int j = k * kThreads + threadIdx.x;
        float z[VW];
        if (j < nv) {
          E::unpack(load_vec<DT, VEC>(rowd, v0, v1, j), z);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) z[e] = neg_inf();
        }
        const int32_t base = static_cast<int32_t>(v0) + j * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const int32_t vi = base + e;
          const bool pass = j < nv && vi < v1 && vi != excl && (!bounded || z[e] >= thr) &&
                            key_beats(z[e], vi, L.tv, L.ti);
          unsigned mm = __ballot_sync(0xffffffffu, pass);
          while (mm) {
            const int src = __ffs(mm) - 1;
            mm &= mm - 1;
            const float zz = __shfl_sync(0xffffffffu, z[e], src);
            const int32_t jj = __shfl_sync(0xffffffffu, vi, src);
            L.insert(zz, jj, F, lane);
          }
        }
      }
      if (lane < F) {
        wl_v[warp][lane] = L.v;
        wl_i[warp][lane] = L.i;
      }
      __syncthreads();
      if (warp == 0) merge_lists(wl_v, wl_i, kWarps, F, lane, outv, outi);
    }
  }
}

}  // namespace specv
