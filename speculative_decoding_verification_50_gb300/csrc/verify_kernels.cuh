// Verification kernels: a1 row statistics, a2 accept test, a3 residual/bonus
// draw ("Speculative Speculative Decoding" §2.1; "Speculative Decoding"
// dl-note §2.2-§2.3; "Lecture 5 - Speculative Decoding and SpecInfer" §2.2,
// §2.7, §3.1).
//
// Work decomposition.  A *unit* is one (batch row b, position i), i in [0, K]:
// for i < K the pair (target row i, draft row i), for i = K the target row K
// alone.  Each unit is owned by a thread-block cluster of C CTAs; CTA `rank`
// owns the vocabulary slice [rank*L, min(V, (rank+1)*L)).
//
//   phase 1  every CTA streams its slice of both rows once from HBM with
//            16-byte loads and keeps an online (max, sum 2^((z-max)*log2e/T))
//            per row (greedy rows: first argmax); block reduction.
//   exchange CTAs publish their partials in shared memory; after a cluster
//            barrier every CTA reads all C partials through distributed
//            shared memory and combines them in rank order, so all CTAs hold
//            bit-identical row statistics.
//   decide   every CTA evaluates the accept test of position i itself
//            (u_i <= p_i(x_i)/q_i(x_i), two scalar loads), so the branch that
//            follows is uniform across the cluster.
//   phase 3  only when position i is rejected (or i = K) does the cluster
//            form r = max(p_i - q_i, 0) (or p_K) over its slices -- a re-read
//            of data this CTA streamed microseconds earlier -- and reduce it
//            to per-warp segment sums; a second exchange gives every CTA the
//            per-CTA totals, hence R and the CTA whose range holds U_K * R;
//            that CTA walks its segments and one warp scans the one segment
//            that holds the crossing.
//   finalize one thread per batch row picks n = the first rejected position
//            and writes the outputs (verify_finalize_kernel).
//
// Every position's bonus candidate is computed speculatively, because the
// first rejection is only known once all positions are decided; accepted
// positions skip phase 3 entirely.
#pragma once

#include <climits>

#include "specv_common.cuh"

namespace specv {

struct UnitOut {      // per (b, i) result, 32 bytes
  int32_t accept;     // 1: draft token x_i accepted (i < K)
  int32_t token;      // bonus candidate t*_i, or -1 when not needed
  float p;            // p_i(x_i)
  float q;            // q_i(x_i)
  int32_t status;     // row-status bits seen by this unit
  int32_t pad[3];
};
static_assert(sizeof(UnitOut) == 32, "UnitOut layout");

struct VerifyParams {
  const void* zt;
  int64_t t_bs, t_rs;
  const void* zd;
  int64_t d_bs, d_rs;
  const int32_t* tokens;
  const float* temp;
  const float* unif;
  UnitOut* units;
  int32_t B, K, V, C, L;
};

// Partial row statistics one CTA publishes to its cluster.
struct Part {
  float mt, st, md, sd;  // temperature rows: running max, sum of 2^((z-m)c)
  float bt, bd;          // greedy rows: best logit
  int32_t it, id;        // greedy rows: first index of the best logit
  int32_t bad;           // greedy rows: NaN or +inf seen
};

// Online (max, sum) over a thread's logits, VW partial sums for accuracy.
template <int VW>
struct Soft {
  float m;
  float s[VW];
  __device__ __forceinline__ void init() {
    m = kNegMax;
#pragma unroll
    for (int k = 0; k < VW; ++k) s[k] = 0.f;
  }
  __device__ __forceinline__ void add(const float (&z)[VW], float c) {
    float vm = z[0];
#pragma unroll
    for (int k = 1; k < VW; ++k) vm = fmaxf(vm, z[k]);  // NaN ignored here
    if (vm > m) {
      const float f = ex2((m - vm) * c);
#pragma unroll
      for (int k = 0; k < VW; ++k) s[k] *= f;
      m = vm;
    }
#pragma unroll
    for (int k = 0; k < VW; ++k) s[k] += ex2((z[k] - m) * c);  // NaN -> sum NaN
  }
  __device__ __forceinline__ float total() const {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < VW; ++k) t += s[k];
    return t;
  }
};

__device__ __forceinline__ void soft_merge(float& m, float& s, float m2, float s2, float c) {
  const float M = fmaxf(m, m2);
  s = s * ex2((m - M) * c) + s2 * ex2((m2 - M) * c);
  m = M;
}

// First argmax over a thread's logits.
struct Arg {
  float best;
  int32_t idx;
  int32_t bad;
  __device__ __forceinline__ void init() {
    best = neg_inf();
    idx = INT_MAX;
    bad = 0;
  }
  template <int VW>
  __device__ __forceinline__ void add(const float (&z)[VW], int32_t base) {
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      bad |= !(z[k] < pos_inf());  // NaN or +inf
      if (z[k] > best) {
        best = z[k];
        idx = base + k;
      }
    }
  }
  __device__ __forceinline__ void merge(float b2, int32_t i2, int32_t bad2) {
    if (b2 > best || (b2 == best && i2 < idx)) {
      best = b2;
      idx = i2;
    }
    bad |= bad2;
  }
};

// Phase 1 over the CTA's slice: vectors j = tid, tid + 256, ... of both rows,
// four vectors per row in flight per thread.
template <int DT, bool VEC, bool GREEDY>
__device__ __forceinline__ void phase1(const void* rowt, const void* rowd, bool pair,
                                       int64_t v0, int64_t v1, int nv, float c,
                                       Soft<Elem<DT>::VW>& st, Soft<Elem<DT>::VW>& sd,
                                       Arg& at, Arg& ad) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  constexpr int U = 4;
  for (int j0 = threadIdx.x; j0 < nv; j0 += U * kThreads) {
    typename E::Vec wt[U], wd[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * kThreads;
      if (j < nv) {
        wt[u] = load_vec<DT, VEC>(rowt, v0, v1, j);
        if (pair) wd[u] = load_vec<DT, VEC>(rowd, v0, v1, j);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * kThreads;
      if (j < nv) {
        float z[VW];
        E::unpack(wt[u], z);
        const int32_t base = static_cast<int32_t>(v0) + j * VW;
        if (GREEDY) at.add(z, base); else st.add(z, c);
        if (pair) {
          E::unpack(wd[u], z);
          if (GREEDY) ad.add(z, base); else sd.add(z, c);
        }
      }
    }
  }
}

// r values of vector j: mode 0 residual max(p - q, 0), mode 1 target p.
template <int DT, bool VEC>
__device__ __forceinline__ void residual_vec(const void* rowt, const void* rowd, int64_t v0,
                                             int64_t v1, int j, int mode, float mt, float md,
                                             float c, float ist, float isd,
                                             float (&r)[Elem<DT>::VW]) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  float zt[VW];
  E::unpack(load_vec<DT, VEC>(rowt, v0, v1, j), zt);
  if (mode == 0) {
    float zd[VW];
    E::unpack(load_vec<DT, VEC>(rowd, v0, v1, j), zd);
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      // Both products rounded before the subtraction (no FMA contraction), so
      // p(v) = q(v) gives r(v) = 0 exactly, as in the definition.
      const float p = __fmul_rn(ex2((zt[k] - mt) * c), ist);
      const float q = __fmul_rn(ex2((zd[k] - md) * c), isd);
      r[k] = fmaxf(__fsub_rn(p, q), 0.f);
    }
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) r[k] = ex2((zt[k] - mt) * c) * ist;
  }
}

// Per-unit decision, computed once by thread 0 and broadcast through shared
// memory (fp64 is a slow path on this GPU; no thread but one touches it).
struct Decision {
  float mt, md, c, ist, isd, px, qx;
  int32_t status, accept, need_scan, token, mode, owner, last_pos;
  double tau, pre_mine;
};

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) verify_units_kernel(const VerifyParams P) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  extern __shared__ float segs[];  // [tiles * kWarps] segment sums of r
  __shared__ Part warp_part[kWarps];
  __shared__ Part cta_part;
  __shared__ double cta_total;
  __shared__ Decision dec;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = P.C;
  const int64_t u = blockIdx.x / C;
  const int K = P.K;
  const int b = static_cast<int>(u / (K + 1));
  const int i = static_cast<int>(u % (K + 1));
  const bool pair = i < K;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const float T = P.temp[b];
  const bool greedy = (T == 0.f);
  const bool temp_ok = (T >= 0.f && T < pos_inf());
  // log2(e)/T (fp32, correctly rounded division).
  const float c = (greedy || !temp_ok) ? 1.f : __fdiv_rn(1.44269504088896341f, T);
  const int x = pair ? P.tokens[static_cast<int64_t>(b) * K + i] : -1;

  const void* rowt = static_cast<const char*>(P.zt) +
                     (static_cast<int64_t>(b) * P.t_bs + static_cast<int64_t>(i) * P.t_rs) * E::ES;
  const void* rowd = pair ? static_cast<const char*>(P.zd) +
                                (static_cast<int64_t>(b) * P.d_bs + static_cast<int64_t>(i) * P.d_rs) * E::ES
                          : rowt;
  const int64_t v0 = static_cast<int64_t>(rank) * P.L;
  const int64_t v1 = min(static_cast<int64_t>(P.V), v0 + P.L);
  const int nv = v1 > v0 ? static_cast<int>((v1 - v0 + VW - 1) / VW) : 0;
  const int ntl = (nv + kThreads - 1) / kThreads;

  // ---- phase 1: row statistics over this CTA's slice ----------------------
  Soft<VW> st, sd;
  Arg at, ad;
  st.init();
  sd.init();
  at.init();
  ad.init();
  if (greedy) phase1<DT, VEC, true>(rowt, rowd, pair, v0, v1, nv, c, st, sd, at, ad);
  else phase1<DT, VEC, false>(rowt, rowd, pair, v0, v1, nv, c, st, sd, at, ad);
  {
    float mt = st.m, s_t = st.total(), md = sd.m, s_d = sd.total();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float mt2 = __shfl_xor_sync(0xffffffffu, mt, o);
      const float st2 = __shfl_xor_sync(0xffffffffu, s_t, o);
      const float md2 = __shfl_xor_sync(0xffffffffu, md, o);
      const float sd2 = __shfl_xor_sync(0xffffffffu, s_d, o);
      const float bt2 = __shfl_xor_sync(0xffffffffu, at.best, o);
      const int it2 = __shfl_xor_sync(0xffffffffu, at.idx, o);
      const int badt2 = __shfl_xor_sync(0xffffffffu, at.bad, o);
      const float bd2 = __shfl_xor_sync(0xffffffffu, ad.best, o);
      const int id2 = __shfl_xor_sync(0xffffffffu, ad.idx, o);
      const int badd2 = __shfl_xor_sync(0xffffffffu, ad.bad, o);
      soft_merge(mt, s_t, mt2, st2, c);
      soft_merge(md, s_d, md2, sd2, c);
      at.merge(bt2, it2, badt2);
      ad.merge(bd2, id2, badd2);
    }
    if (lane == 0) {
      Part& w = warp_part[warp];
      w.mt = mt; w.st = s_t; w.md = md; w.sd = s_d;
      w.bt = at.best; w.it = at.idx; w.bd = ad.best; w.id = ad.idx;
      w.bad = at.bad | ad.bad;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Part p = warp_part[0];
    Arg gt, gd;
    gt.best = p.bt; gt.idx = p.it; gt.bad = p.bad;
    gd.best = p.bd; gd.idx = p.id; gd.bad = 0;
    for (int w = 1; w < kWarps; ++w) {
      const Part& q = warp_part[w];
      soft_merge(p.mt, p.st, q.mt, q.st, c);
      soft_merge(p.md, p.sd, q.md, q.sd, c);
      gt.merge(q.bt, q.it, q.bad);
      gd.merge(q.bd, q.id, 0);
    }
    p.bt = gt.best; p.it = gt.idx; p.bd = gd.best; p.id = gd.idx; p.bad = gt.bad;
    cta_part = p;
  }
  cluster.sync();  // (1) partials visible cluster-wide

  // ---- exchange + decide (thread 0; identical in every CTA) ---------------
  double St = 0.0, Sd = 0.0;  // live in thread 0 only
  if (threadIdx.x == 0) {
    int status = temp_ok ? 0 : kBadTemp;
    if (pair && (x < 0 || x >= P.V)) status |= kBadToken;
    float Mt = kNegMax, Md = kNegMax;
    Arg gt, gd;
    gt.init();
    gd.init();
    for (int r = 0; r < C; ++r) {
      const Part* q = cluster.map_shared_rank(&cta_part, r);
      Mt = fmaxf(Mt, q->mt);
      Md = fmaxf(Md, q->md);
      gt.merge(q->bt, q->it, q->bad);
      gd.merge(q->bd, q->id, 0);
    }
    for (int r = 0; r < C; ++r) {
      const Part* q = cluster.map_shared_rank(&cta_part, r);
      St += static_cast<double>(q->st) * static_cast<double>(ex2((q->mt - Mt) * c));
      Sd += static_cast<double>(q->sd) * static_cast<double>(ex2((q->md - Md) * c));
    }
    if (temp_ok) {
      if (greedy) {
        if (gt.bad || gt.idx == INT_MAX || (pair && gd.idx == INT_MAX)) status |= kNonFinite;
      } else {
        if (!(St >= 1.0) || Mt == kNegMax) status |= kNonFinite;
        if (pair && (!(Sd >= 1.0) || Md == kNegMax)) status |= kNonFinite;
      }
    }
    int accept = 0;
    float px = 0.f, qx = 0.f;
    if (pair && !(status & kErrors)) {
      if (greedy) {
        px = (x == gt.idx) ? 1.f : 0.f;
        qx = (x == gd.idx) ? 1.f : 0.f;
        accept = (x == gt.idx) && (x == gd.idx);
      } else {
        const float ztx = E::scalar(rowt, x);
        const float zdx = E::scalar(rowd, x);
        const float lt = __fmul_rn(ztx - Mt, c);  // log2 of unnormalised p_i(x), q_i(x)
        const float ld = __fmul_rn(zdx - Md, c);
        px = static_cast<float>(static_cast<double>(ex2(lt)) / St);
        qx = static_cast<float>(static_cast<double>(ex2(ld)) / Sd);
        if (zdx != neg_inf()) {  // q_i(x_i) > 0
          const double ratio = static_cast<double>(ex2(__fsub_rn(lt, ld))) * (Sd / St);
          accept = ratio >= static_cast<double>(P.unif[static_cast<int64_t>(b) * (K + 1) + i]);
        }
      }
    }
    const bool need_bonus = !(status & kErrors) && !(pair && accept);
    dec.mt = Mt;
    dec.md = Md;
    dec.c = c;
    dec.ist = static_cast<float>(1.0 / St);
    dec.isd = static_cast<float>(1.0 / Sd);
    dec.px = px;
    dec.qx = qx;
    dec.status = status;
    dec.accept = accept;
    dec.need_scan = need_bonus && !greedy;
    dec.token = (need_bonus && greedy) ? gt.idx : -1;
    dec.mode = pair ? 0 : 1;
    dec.owner = -1;
    dec.last_pos = 0;
    dec.tau = 0.0;
    dec.pre_mine = 0.0;
  }
  __syncthreads();

  if (dec.need_scan) {
    // ---- phase 3: residual (or target) mass, per-warp segment sums --------
    for (int attempt = 0; attempt < 2; ++attempt) {
      const int mode = dec.mode;
      const float mt = dec.mt, md = dec.md, ist = dec.ist, isd = dec.isd;
      for (int t = 0; t < ntl; t += 2) {
        const int j0 = t * kThreads + threadIdx.x;
        const int j1 = j0 + kThreads;
        float r0[VW], r1[VW];
        float s0 = 0.f, s1 = 0.f;
        if (j0 < nv) residual_vec<DT, VEC>(rowt, rowd, v0, v1, j0, mode, mt, md, c, ist, isd, r0);
        if (j1 < nv) residual_vec<DT, VEC>(rowt, rowd, v0, v1, j1, mode, mt, md, c, ist, isd, r1);
        if (j0 < nv) {
#pragma unroll
          for (int k = 0; k < VW; ++k) s0 += r0[k];
        }
        if (j1 < nv) {
#pragma unroll
          for (int k = 0; k < VW; ++k) s1 += r1[k];
        }
        s0 = warp_sum(s0);
        s1 = warp_sum(s1);
        if (lane == 0) {
          segs[t * kWarps + warp] = s0;
          if (t + 1 < ntl) segs[(t + 1) * kWarps + warp] = s1;
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int s = 0; s < ntl * kWarps; ++s) tot += static_cast<double>(segs[s]);
        cta_total = tot;
      }
      cluster.sync();  // (2) per-CTA totals visible
      if (threadIdx.x == 0) {
        double R = 0.0;
        int last_rank = -1;
        for (int r = 0; r < C; ++r) {
          const double tr = *cluster.map_shared_rank(&cta_total, r);
          if (r == rank) dec.pre_mine = R;
          if (tr > 0.0) last_rank = r;
          R += tr;
        }
        const double tau = static_cast<double>(P.unif[static_cast<int64_t>(b) * (K + 1) + K]) * R;
        int owner = -1;
        double pre = 0.0;
        for (int r = 0; r < C; ++r) {
          const double tr = *cluster.map_shared_rank(&cta_total, r);
          if (owner < 0 && tr > 0.0 && pre + tr > tau) owner = r;
          pre += tr;
        }
        dec.tau = tau;
        if (R > 0.0) {
          if (owner < 0) {  // U*R >= R after rounding: last index with r > 0
            owner = last_rank;
            dec.last_pos = 1;
            dec.status |= kFallback;
          }
          dec.owner = owner;
        } else if (dec.mode == 0) {
          dec.mode = 1;  // zero residual mass: draw from p_i instead
          dec.status |= kFallback;
        }
      }
      cluster.sync();  // (3) totals read by everyone; dec visible in the CTA
      if (dec.owner >= 0 || dec.mode == 0 || attempt == 1) break;
    }

    // ---- owner CTA: locate the crossing segment, then scan it --------------
    if (rank == dec.owner && warp == 0) {
      const int nseg = ntl * kWarps;
      const double tau = dec.tau;
      int seg = -1, lastseg = -1;
      double cum_at = 0.0;
      if (lane == 0) {
        double cum = dec.pre_mine;
        for (int s = 0; s < nseg; ++s) {
          const float g = segs[s];
          if (g > 0.f) {
            if (seg < 0 && !dec.last_pos && cum + static_cast<double>(g) > tau) {
              seg = s;
              cum_at = cum;
            }
            lastseg = s;
            cum += static_cast<double>(g);
          }
        }
      }
      seg = __shfl_sync(0xffffffffu, seg, 0);
      lastseg = __shfl_sync(0xffffffffu, lastseg, 0);
      cum_at = __shfl_sync(0xffffffffu, cum_at, 0);
      bool lp = dec.last_pos || seg < 0;
      if (seg < 0) seg = lastseg;
      const int j = (seg / kWarps) * kThreads + (seg % kWarps) * 32 + lane;
      float r[VW];
#pragma unroll
      for (int k = 0; k < VW; ++k) r[k] = 0.f;
      if (seg >= 0 && j < nv)
        residual_vec<DT, VEC>(rowt, rowd, v0, v1, j, dec.mode, dec.mt, dec.md, c, dec.ist,
                              dec.isd, r);
      const int32_t base = static_cast<int32_t>(v0) + j * VW;
      int found = -1;  // token found by this lane
      if (!lp) {
        float vs = 0.f;
#pragma unroll
        for (int k = 0; k < VW; ++k) vs += r[k];
        double incl = static_cast<double>(vs);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const double excl = incl - static_cast<double>(vs);
        const unsigned m = __ballot_sync(0xffffffffu, vs > 0.f && cum_at + incl > tau);
        if (m) {
          if (lane == __ffs(m) - 1) {
            double run = cum_at + excl;
            int kk = -1, klast = -1;
#pragma unroll
            for (int k = 0; k < VW; ++k) {
              if (r[k] > 0.f) {
                run += static_cast<double>(r[k]);
                klast = k;
                if (kk < 0 && run > tau) kk = k;
              }
            }
            found = base + (kk >= 0 ? kk : klast);
          }
        } else {
          lp = true;
        }
      }
      if (lp) {
        int kl = -1;
#pragma unroll
        for (int k = 0; k < VW; ++k)
          if (r[k] > 0.f) kl = k;
        const unsigned m = __ballot_sync(0xffffffffu, kl >= 0);
        if (m && lane == 31 - __clz(m)) found = base + kl;
      }
      const unsigned mf = __ballot_sync(0xffffffffu, found >= 0);
      const int tok = mf ? __shfl_sync(0xffffffffu, found, __ffs(mf) - 1) : -1;
      if (lane == 0) dec.token = tok;
    }
  } else {
    cluster.sync();  // (2') no CTA exits while a peer may read its partials
  }

  // Exactly one CTA writes the unit's result.
  const int writer = (dec.need_scan && dec.owner >= 0) ? dec.owner : 0;
  if (rank == writer && threadIdx.x == 0) {
    UnitOut& o = P.units[u];
    o.accept = dec.accept;
    o.token = dec.token;
    o.p = dec.px;
    o.q = dec.qx;
    o.status = dec.status;
  }
}

// Per batch row: accept length = first rejected position; tokens; outputs.
__global__ void verify_finalize_kernel(const UnitOut* __restrict__ units,
                                       const int32_t* __restrict__ tokens, int B, int K,
                                       int32_t* __restrict__ accept_len,
                                       int32_t* __restrict__ out_tokens,
                                       float* __restrict__ p_draft, float* __restrict__ q_draft,
                                       int32_t* __restrict__ row_status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const UnitOut* U = units + static_cast<int64_t>(b) * (K + 1);
  int err = 0;
  for (int i = 0; i <= K; ++i) err |= U[i].status & kErrors;
  int32_t* ot = out_tokens + static_cast<int64_t>(b) * (K + 1);
  if (err) {
    accept_len[b] = 0;
    for (int i = 0; i <= K; ++i) ot[i] = -1;
    if (p_draft)
      for (int i = 0; i < K; ++i) p_draft[static_cast<int64_t>(b) * K + i] = 0.f;
    if (q_draft)
      for (int i = 0; i < K; ++i) q_draft[static_cast<int64_t>(b) * K + i] = 0.f;
    if (row_status) row_status[b] = err;
    return;
  }
  int n = K;
  for (int i = 0; i < K; ++i)
    if (!U[i].accept) {
      n = i;
      break;
    }
  accept_len[b] = n;
  for (int i = 0; i < n; ++i) ot[i] = tokens[static_cast<int64_t>(b) * K + i];
  ot[n] = U[n].token;
  for (int i = n + 1; i <= K; ++i) ot[i] = -1;
  if (p_draft)
    for (int i = 0; i < K; ++i) p_draft[static_cast<int64_t>(b) * K + i] = U[i].p;
  if (q_draft)
    for (int i = 0; i < K; ++i) q_draft[static_cast<int64_t>(b) * K + i] = U[i].q;
  if (row_status) row_status[b] = U[n].status & kFallback;
}

}  // namespace specv
