// Kernel B of the hot path: per batch row, from kernel A's chunk records,
//   a2 the left-to-right accept test u_i <= p_i(x_i)/q_i(x_i) up to the first
//      rejection n ("Lecture 5 - Speculative Decoding and SpecInfer" §2.2,
//      §2.7; "Speculative Decoding" dl-note Appendix: draft prob 0 rejects),
//   a3 the bonus t* by inverse CDF of r = max(p_n - q_n, 0), or of p_K when
//      all K drafts are accepted ("Speculative Speculative Decoding" §2.1;
//      dl-note §2.3; Lecture 5 §3.1),
//   a4 the outcome keys: top-F of the per-chunk candidates at each lookahead
//      ("Speculative Speculative Decoding" §4.1.1), and
//   a5 the hit flag: t* among the keys of lookahead n (§3.1);
// in its other modes the Saguaro sampler's draw from sigma_{F,C} (§4.2.1)
// and multi-step speculative sampling at token-tree nodes (Lecture 5 §6.4).
//
// One thread-block cluster of CB CTAs per batch row.  Every CTA combines the
// records itself (half a warp per position, lanes over chunks, float-float
// sums) and decides n; the arithmetic and its order are the same everywhere,
// so all CTAs agree without waiting for one another.  Only row n is read
// again: every CTA streams its slice of target row n (and draft row n) through
// a bulk-copy ring, forms r, and reduces it to per-warp segment sums; the
// per-CTA totals are exchanged through distributed shared memory, which gives
// R and the CTA whose range holds U_K * R; that CTA walks its segments and one
// warp scans the one segment that holds the crossing (a re-read of 32
// vectors).  A draw from a whole row's own distribution reads only the chunk
// (or, for the sampler, the piece of a chunk) holding U * R instead.
// Meanwhile warps 1..7 of every CTA merge the chunk candidate lists into the
// outcome keys (one warp per lookahead).  Rank 0 writes the outputs.
#pragma once

#include "stats_kernel.cuh"

namespace specv {

constexpr int kTileUnroll = 8;  // tiles of r per loop trip in the residual pass

struct PosStats {  // one position's combined row statistics
  FF St, Sd;  // softmax normalisers, in units of 2^((z - M) c)
  float Mt, Md;
  int32_t it, id;
  int32_t bad;
  int32_t pad;
};

struct Dec {  // a batch row's decision (the same in every CTA of its cluster)
  int32_t n, status, mode, need_scan, token, owner, last_pos, xn;
  float mt, md, ist, isd;
  float sgc, zl;  // residual weights: C on the keys at or above (zl, il)
  int32_t il;
  int32_t full_pass;  // a chunk-local draw reads the whole row instead (see below)
  float zx;      // without draft probabilities: the target logit of the rejected token
  FF R;          // total residual mass (the sampler normalises its q by it)
  FF tau, pre_mine;
  float px[kMaxK], qx[kMaxK];
  // MSS at a token-tree node: the residual after j rejections is
  // max(0, p - c_j q) / D_j with c_0 = 0, D_0 = 1, c_{j+1} = c_j + D_j and
  // D_j = sum_v max(0, p - c_j q) (one pass over the node's rows each).
  FF cff;        // c_j of the current pass
  float cq;      // c_j as a float (the residual's multiplier of q)
  int32_t next;  // the candidate tested after the current pass
  int32_t acc;   // the accepted candidate, or -1
  int32_t again; // another pass is needed
  float ap[kMaxK];  // min(1, p_j(x_j)/q(x_j)) of the tested candidates
};
static_assert(sizeof(Dec) % 4 == 0, "Dec copied as words");

struct DecideParams {
  const void* zt;
  int64_t t_bs, t_rs;
  const void* zd;
  int64_t d_bs, d_rs;
  const int32_t* tokens;
  const float* temp;
  const float* unif;
  const ChunkRec* recs;
  const float* cand_v;
  const int32_t* cand_i;
  int32_t* accept_len;
  int32_t* out_tokens;
  float* p_draft;
  float* q_draft;
  int32_t* row_status;
  int32_t* keys;
  float* key_logits;
  uint8_t* hit;
  int32_t B, K, V, F, nchunk, CB, L;
  int32_t chunk;     // logits per chunk record of the row-statistics kernel
  int32_t fk[kMaxK + 1];  // keys kept at lookahead k (F when the fan-out is uniform)
  int32_t stages;    // ring stages of the staged residual pass (aligned rows); 0: none
  int32_t ring_off;  // byte offset of that ring in dynamic shared memory
  const int32_t* cu; // per-row draft counts (inclusive prefix sums), or null
  int32_t ntok;      // with cu: packed draft rows the buffers hold
  int32_t no_draft;  // no draft logits: q_i is one-hot at x_i
  int32_t sg_F;      // Saguaro sampling: the drafts came from sigma_{sg_F, sg_C}
  float sg_C;        //   (0: plain softmax drafts); the sampler's own F and C
  int32_t local_draw;  // draws from a whole row read only the chunk holding U * R
  int32_t pieces;      // the sampler's chunks are split in pieces (2, 4 or 8; 0: none)
  const float2* piece_stats;  // their (max, sum), kMaxPieces entries per chunk
  int32_t stall;       // test hook: 1 + the batch row whose first residual stage (rank 0)
                       // waits for 16 bytes no copy brings, so its wait runs out (0: none)
  // MSS (K = M candidates per node, one target and one draft row each)
  const int32_t* ncand;  // per-node candidate counts, or null (all M)
  int32_t naive;         // naive sampling: one draw from p, candidates matched to it
  int32_t* mss_acc;      // [B] accepted candidate or -1
  float* mss_ap;         // optional [B, M] accept probabilities
};

// Combine the chunk records of one position over an aligned group of W lanes
// (`sub` = lane within the group; result in every lane of the group).
template <int W>
__device__ __forceinline__ PosStats combine_position(const ChunkRec* R, int nchunk, float c, int sub) {
  float mt = kNegMax, s_t = 0.f, md = kNegMax, s_d = 0.f;
  Arg at, ad;
  at.init();
  ad.init();
  for (int q = sub; q < nchunk; q += W) {
    const ChunkRec r = ld_rec(R + q);
    soft_merge(mt, s_t, r.mt, r.st, c);
    soft_merge(md, s_d, r.md, r.sd, c);
    at.merge(r.bt, r.it, r.bad);
    ad.merge(r.bd, r.id, 0);
  }
  PosStats p;
  p.Mt = warp_max_all<float, W>(mt);
  p.Md = warp_max_all<float, W>(md);
  p.St = warp_ffsum_all<W>(ff_mul(s_t, ex2((mt - p.Mt) * c)));
  p.Sd = warp_ffsum_all<W>(ff_mul(s_d, ex2((md - p.Md) * c)));
  warp_arg_all<W>(at.best, at.idx);
  warp_arg_all<W>(ad.best, ad.idx);
  p.it = at.idx;
  p.id = ad.idx;
  // bad flags of the whole group (OR over W lanes)
  int bad = at.bad;
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) bad |= __shfl_xor_sync(0xffffffffu, bad, o);
  p.bad = bad;
  p.pad = 0;
  return p;
}

// Top-F keys of one draft row from its per-chunk candidate lists, by one warp
// (lanes < F end with the keys of rank `lane`; (-inf, INT_MAX) where the row
// has fewer than F).  Up to kStageCand candidates are staged in the warp's
// shared scratch and merged by the lists' heads (or ranked by counting when
// there are more lists than lanes); larger sets are merged by warp
// insertion.  The sampler's CTA ranks up to kWarpCand candidates with all
// its threads (four per candidate).
constexpr int kWarpCand = 64;
constexpr int kStageCand = 128;  // a fan-out's widest lookahead: 7 chunks x 16 keys
struct WarpKeys {
  float v[kStageCand];
  int32_t i[kStageCand];
  float ov[kMaxF];
  int32_t oi[kMaxF];
};

__device__ __forceinline__ WarpTopF merge_candidates(const float* cv, const int32_t* ci, int ncand,
                                                     int F, int lane);

// nkeep <= F: only the first nkeep keys are wanted (a fan-out's lookahead).
__device__ __forceinline__ WarpTopF warp_keys(const float* cv, const int32_t* ci, int ncand, int F,
                                              int lane, WarpKeys& S, int nkeep = kMaxF) {
  if (ncand > kStageCand) return merge_candidates(cv, ci, ncand, F, lane);
  for (int e = lane; e < ncand; e += 32) {
    S.v[e] = __ldcg(cv + e);
    S.i[e] = __ldcg(ci + e);
  }
  __syncwarp();
  WarpTopF L;
  L.init();
  const int nl = ncand / F;  // the chunks' lists, F entries each in key order
  if (nl <= 32) {
    // merge by their heads: lane l follows list l; F rounds of a warp
    // argmax, the winning lane stepping to its list's next entry (indices are
    // distinct across chunks; empty entries (-inf, INT_MAX) come last)
    int ptr = 0;
    float hv = neg_inf();
    int32_t hi = INT_MAX;
    if (lane < nl) {
      hv = S.v[lane * F];
      hi = S.i[lane * F];
    }
    const int rounds = min(F, nkeep);
    for (int f = 0; f < rounds; ++f) {
      float bv = hv;
      int32_t bi = hi;
      int bl = lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
        const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
        if (key_beats(ov, oi, bv, bi) || (ov == bv && oi == bi && ol < bl)) {
          bv = ov;
          bi = oi;
          bl = ol;
        }
      }
      if (lane == f) {
        L.v = bv;
        L.i = bi;
      }
      if (lane == bl && bi != INT_MAX) {
        ++ptr;
        hv = ptr < F ? S.v[lane * F + ptr] : neg_inf();
        hi = ptr < F ? S.i[lane * F + ptr] : INT_MAX;
      }
    }
    __syncwarp();  // the scratch may be reused by this warp's next row
    return L;
  }
  // more lists than lanes: rank every candidate by counting
  if (lane < F) {
    S.ov[lane] = neg_inf();
    S.oi[lane] = INT_MAX;
  }
  __syncwarp();
  for (int e = lane; e < ncand; e += 32) {
    const float v = S.v[e];
    const int32_t i = S.i[e];
    if (i == INT_MAX) continue;  // an empty slot of a short list
    int rank = 0;
    for (int o = 0; o < ncand; ++o) rank += key_beats(S.v[o], S.i[o], v, i);
    if (rank < F) {
      S.ov[rank] = v;
      S.oi[rank] = i;
    }
  }
  __syncwarp();
  if (lane < F) {
    L.v = S.ov[lane];
    L.i = S.oi[lane];
  }
  __syncwarp();  // the scratch may be reused by this warp's next row
  return L;
}

// The same ranking with the whole CTA (the sampler's one row): four threads
// per candidate, each counting the candidates that beat it in a quarter of
// the list.  ncand <= kWarpCand; the top F land in S.ov / S.oi.
static_assert(kThreads == 4 * kWarpCand, "four threads per candidate");
__device__ __forceinline__ void cta_rank_keys(const float* cv, const int32_t* ci, int ncand, int F,
                                              WarpKeys& S) {
  const int t = threadIdx.x;
  if (t < ncand) {
    S.v[t] = __ldcg(cv + t);
    S.i[t] = __ldcg(ci + t);
  }
  if (t < F) {
    S.ov[t] = neg_inf();
    S.oi[t] = INT_MAX;
  }
  __syncthreads();
  const int e = t >> 2, o0 = (t & 3) * (kWarpCand / 4), o1 = min(ncand, o0 + kWarpCand / 4);
  float v = neg_inf();
  int32_t i = INT_MAX;
  int rank = 0;
  if (e < ncand) {
    v = S.v[e];
    i = S.i[e];
    for (int o = o0; o < o1; ++o) rank += key_beats(S.v[o], S.i[o], v, i);
  }
  rank += __shfl_xor_sync(0xffffffffu, rank, 1);
  rank += __shfl_xor_sync(0xffffffffu, rank, 2);
  if ((t & 3) == 0 && e < ncand && i != INT_MAX && rank < F) {
    S.ov[rank] = v;
    S.oi[rank] = i;
  }
  __syncthreads();
}

// Top-F over the per-chunk candidate lists of one draft row (warp-wide).
__device__ __forceinline__ WarpTopF merge_candidates(const float* cv, const int32_t* ci, int ncand,
                                                     int F, int lane) {
  WarpTopF L;
  L.init();
  for (int base = 0; base < ncand; base += 32) {
    const int idx = base + lane;
    float z = neg_inf();
    int32_t vi = INT_MAX;
    if (idx < ncand) {
      z = __ldcg(cv + idx);
      vi = __ldcg(ci + idx);
    }
    unsigned m = __ballot_sync(0xffffffffu, vi != INT_MAX && key_beats(z, vi, L.tv, L.ti));
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const float zz = __shfl_sync(0xffffffffu, z, src);
      const int32_t ii = __shfl_sync(0xffffffffu, vi, src);
      L.insert(zz, ii, F, lane);
    }
  }
  return L;
}

// r values of one vector (logits e0 .. e0+VW-1) from its target (and draft)
// logits: mode 0 max(p - q, 0); mode 1 p; mode 2 (no draft probabilities: q
// one-hot at the rejected token xn) p with r(xn) = 0.  Both products rounded
// before the subtraction (no contraction), so p(v) = q(v) gives r(v) = 0
// exactly, as in the definition.
// Saguaro weights ([SSD] §4.2.1): a logit z at index e is among the row's
// top-F_s, and is weighted by C, iff its key (z, e) is at or above the F_s-th
// key (zl, il) in (logit desc, index asc) order.  zl = +inf: no weights.
struct SgW {
  float C, zl;
  int32_t il;
  __device__ __forceinline__ bool in(float z, int64_t e) const {
    return z > zl || (z == zl && e <= il);
  }
};

template <int VW>
__device__ __forceinline__ void residual_from(const float (&zt)[VW], const float (&zd)[VW], int mode,
                                              float mt, float md, float c, float ist, float isd,
                                              int64_t e0, int xn, const SgW& w, float (&r)[VW]) {
  if (mode == 2) {
#pragma unroll
    for (int k = 0; k < VW; ++k)
      r[k] = (e0 + k == xn) ? 0.f : __fmul_rn(ex2((zt[k] - mt) * c), ist);
  } else if (mode == 3) {  // the sampler: sigma_{F,C} of the row itself
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const float p = __fmul_rn(ex2((zt[k] - mt) * c), ist);
      r[k] = w.in(zt[k], e0 + k) ? __fmul_rn(p, w.C) : p;
    }
  } else if (mode == 0 && w.zl == pos_inf()) {  // plain softmax drafts
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const float p = __fmul_rn(ex2((zt[k] - mt) * c), ist);
      const float q = __fmul_rn(ex2((zd[k] - md) * c), isd);
      r[k] = fmaxf(__fsub_rn(p, q), 0.f);
    }
  } else if (mode == 0) {  // q is sigma_{F,C} of the draft row
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const float p = __fmul_rn(ex2((zt[k] - mt) * c), ist);
      float q = __fmul_rn(ex2((zd[k] - md) * c), isd);
      if (w.in(zd[k], e0 + k)) q = __fmul_rn(q, w.C);
      r[k] = fmaxf(__fsub_rn(p, q), 0.f);
    }
  } else {
#pragma unroll
    for (int k = 0; k < VW; ++k) r[k] = __fmul_rn(ex2((zt[k] - mt) * c), ist);
  }
}

// r values of vector j of a row slice, read from global memory.
template <int DT, bool VEC>
__device__ __forceinline__ void residual_vec(const void* rowt, const void* rowd, int64_t v0,
                                             int64_t v1, int j, int mode, float mt, float md,
                                             float c, float ist, float isd, int xn, const SgW& w,
                                             float (&r)[Elem<DT>::VW]) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  float zt[VW], zd[VW];
  E::unpack(load_vec<DT, VEC>(rowt, v0, v1, j), zt);
  if (mode == 0) E::unpack(load_vec<DT, VEC>(rowd, v0, v1, j), zd);
  residual_from<VW>(zt, zd, mode, mt, md, c, ist, isd, v0 + static_cast<int64_t>(j) * VW, xn, w, r);
}

// Staged residual pass (16-byte aligned rows): the slice C of target row n
// (and draft row n in mode 0) streams through the same bulk-copy ring as the
// row-statistics kernel; trip t holds tiles 2t and 2t+1 (tile = one 16-byte
// vector per thread).  ring_start arms the ring and issues the first trips (by
// thread 0; call before other work, then a CTA barrier); ring_residual
// consumes them and writes the per-warp segment sums of r, tile-major, as the
// register path does.  Returns false if a wait gave up (after a bounded wait
// for the copies still in flight).  With `stall` (a test hook) stage 0 also
// waits for 16 bytes that no copy brings.  `stream`: the copies are marked
// evict-first (a row read once); an MSS node, whose later passes read the
// same two rows again, keeps the default policy.
// Invalidates the ring's barriers, before ring_start arms them for another
// pass (every wait on them has ended and every copy has landed).
__device__ __forceinline__ void ring_reset(RingBars& R, int S) {
  if (threadIdx.x == 0)
    for (int s = 0; s < S; ++s)
      asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&R.full[s])) : "memory");
}

template <int DT>
__device__ __forceinline__ void ring_start(RingBars& R, unsigned char* ring, int S, const Chunk& C,
                                           bool stall = false, bool stream = true) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&R.full[s], 1);
    fence_mbar_init();
    if (stall) mbar_expect_tx(&R.full[0], 16);
    const int ntr = ring_trips(C.nv);
    for (int t = 0; t < ntr && t < S; ++t) ring_issue<DT>(&R.full[t], ring, t, t, C, false, stream);
  }
}

template <int DT>
__device__ __forceinline__ bool ring_residual(RingBars& R, unsigned char* ring, int S, const Chunk& C,
                                              int mode, float mt, float md, float c, float ist,
                                              float isd, int xn, const SgW& w, float* segs, int ntl,
                                              bool stream = true) {
  using E = Elem<DT>;
  using Vec = typename E::Vec;
  constexpr int VW = E::VW;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int ntr = ring_trips(C.nv);
  const int64_t covered = covered_end<DT>(C);
  const int nwhole = whole_trips<DT>(C, covered);
  bool ok = true;
  int s = 0;
  uint32_t ph = 0;
  for (int t = 0; t < ntr; ++t) {
    if (!mbar_wait_bounded(&R.full[s], ph)) ok = false;
    const unsigned char* base = ring + static_cast<int64_t>(s) * 2 * kTripBytes;
    float sum[kVecs];
    if (t < nwhole) {  // whole trip in shared memory: no bounds checks
#pragma unroll
      for (int k = 0; k < kVecs; ++k) {
        const int jl = k * kThreads + threadIdx.x;
        float zt[VW], zd[VW], r[VW];
        E::unpack(reinterpret_cast<const Vec*>(base)[jl], zt);
        if (mode == 0) E::unpack(reinterpret_cast<const Vec*>(base + kTripBytes)[jl], zd);
        const int64_t e0 = C.v0 + static_cast<int64_t>((t * kVecs + k) * kThreads + threadIdx.x) * VW;
        residual_from<VW>(zt, zd, mode, mt, md, c, ist, isd, e0, xn, w, r);
        sum[k] = 0.f;
#pragma unroll
        for (int q = 0; q < VW; ++q) sum[k] += r[q];
      }
    } else {
#pragma unroll
      for (int k = 0; k < kVecs; ++k) {
        const int j = (t * kVecs + k) * kThreads + threadIdx.x;
        sum[k] = 0.f;
        if (j < C.nv) {
          const int64_t e = C.v0 + static_cast<int64_t>(j) * VW;
          const int jl = k * kThreads + threadIdx.x;
          float zt[VW], zd[VW], r[VW];
          if (e + VW <= covered) {
            E::unpack(reinterpret_cast<const Vec*>(base)[jl], zt);
            if (mode == 0) E::unpack(reinterpret_cast<const Vec*>(base + kTripBytes)[jl], zd);
          } else {
            E::unpack(E::gather(C.rowt, e, C.v1), zt);
            if (mode == 0) E::unpack(E::gather(C.rowd, e, C.v1), zd);
          }
          residual_from<VW>(zt, zd, mode, mt, md, c, ist, isd, e, xn, w, r);
#pragma unroll
          for (int q = 0; q < VW; ++q) sum[k] += r[q];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const int tile = t * kVecs + k;
      const float w = warp_sum(sum[k]);
      if (lane == 0 && tile < ntl) segs[tile * kWarps + warp] = w;
    }
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        int s2 = s;
        uint32_t p2 = ph;
        for (int t2 = t; t2 < ntr && t2 < t + S; ++t2) {
          mbar_wait_bounded(&R.full[s2], p2);
          if (++s2 == S) {
            s2 = 0;
            p2 ^= 1u;
          }
        }
      }
      __syncthreads();
      return false;
    }
    if (threadIdx.x == 0 && t + S < ntr) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue<DT>(&R.full[s], ring, s, t + S, C, false, stream);
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  return ok;
}

// Mass of piece p of a sampled row's chunk, in units of 2^((z - M) c), from
// the row-statistics kernel's table (read through L2: another kernel wrote it).
__device__ __forceinline__ FF piece_mass(const float2* stats, int p, float M, float c) {
  const float2 h = __ldcg(stats + p);
  return ff_mul(h.y, ex2((h.x - M) * c));
}

constexpr int kDrawTiles = 16 * kVecs;  // 256-vector tiles in the longest piece read (16 trips)
static_assert(kDrawTiles <= 32, "one lane per tile");

struct DrawSmem {
  float tile[kDrawTiles][kWarps];  // per-warp sums of r in each tile of the chunk
  FF R;        // the row's total mass
  FF tau_in;   // U * R less the mass before the chosen chunk
  float tw;    // U * R less the mass before the chosen warp of the chosen tile
  int32_t pick;    // the chunk, then the token, holding U * R
  int32_t tsel;    // the tile holding it
  int32_t wsel;    // the warp of that tile holding it
  int32_t fallback;
  float q;
};

// A draw from a whole row's own distribution, r(v) = w(v) 2^((z_v - M) c) with
// w = C on the row's top-F_s keys (the sampler) or 1 (the bonus after all K
// drafts are accepted), by inverse CDF of U ("Speculative Speculative
// Decoding" §2.1; §4.2.1); with xex >= 0, w(xex) = 0 (the residual
// max(p - q, 0) when q is one-hot at the rejected token xex, whose logit is
// zex: "Speculative Decoding" dl-note, Appendix, NO_DRAFT_PROBS).  The row-statistics kernel's chunk records give
// every chunk's mass, so the prefix over chunks finds the chunk holding U * R
// and only that chunk is read again: its 256-vector tiles give per-warp sums,
// a scan over tiles and then warps narrows U * R to 32 vectors, and a warp
// scan to one.  Every sum is float-float.  All threads of one CTA call it;
// returns the token, with S.q = r(t) / R and S.fallback set when rounding
// left U * R past the end (the last logit with r > 0 is taken).
template <int DT, bool VEC>
__device__ int chunk_draw(const ChunkRec* recs, int nchunk, int32_t chunk, int V, bool draft_fields,
                          float M, float c, const char* row, float U, const float* kv,
                          const int32_t* ki, int nk, const SgW& w, int pieces,
                          const float2* piece_stats, int32_t xex, float zex, DrawSmem& S) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // With pieces the row-statistics kernel also wrote the statistics of each
  // piece of a chunk (the sampler's chunks): the draw then locates and reads
  // one piece.
  const bool split = pieces > 1;
  const int nloc = split ? pieces * nchunk : nchunk;
  const int32_t span = split ? chunk / pieces : chunk;  // logits per located piece
  // ---- warp 0: chunk masses, lanes over contiguous blocks of chunks --------
  if (warp == 0) {
    const FF one_m_c = two_sum(1.f, -w.C);
    const int per = (nloc + 31) / 32;
    const int j0 = min(nloc, lane * per), j1 = min(nloc, j0 + per);
    auto mass = [&](int j) -> FF {
      FF x;
      if (split) {  // piece j % pieces of chunk j / pieces
        x = piece_mass(piece_stats + static_cast<int64_t>(j / pieces) * kMaxPieces, j % pieces, M, c);
      } else {
        const ChunkRec r = ld_rec(recs + j);
        const float m = draft_fields ? r.md : r.mt, sm = draft_fields ? r.sd : r.st;
        x = ff_mul(sm, ex2((m - M) * c));
      }
      for (int k = 0; k < nk; ++k)  // the weighted keys of this piece
        if (ki[k] / span == j) x = ff_add(x, ff_neg(ff_mul(one_m_c, ex2((kv[k] - M) * c))));
      if (xex >= 0 && xex / span == j) x = ff_add(x, ff(-ex2((zex - M) * c)));  // the excluded token
      return x.hi > 0.f ? x : ff(0.f);
    };
    FF mine = ff(0.f);
    for (int j = j0; j < j1; ++j) mine = ff_add(mine, mass(j));
    const FF incl = warp_ffscan(mine, lane);
    const FF R = shfl(incl, 31);
    const FF tau = ff_mul(R, U);
    const unsigned hit = __ballot_sync(0xffffffffu, mine.hi > 0.f && ff_gt(incl, tau));
    const unsigned pos = __ballot_sync(0xffffffffu, mine.hi > 0.f);
    const bool last = hit == 0;  // U * R at or past the end after rounding
    const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == 0) {
      S.pick = -1;
      S.R = R;
      S.fallback = last ? 1 : 0;
    }
    __syncwarp();
    if (lane == owner) {
      FF run = ff_add(incl, ff_neg(mine));
      int pick = -1;
      FF tin = ff(0.f);
      for (int j = j0; j < j1; ++j) {
        const FF x = mass(j);
        if (x.hi > 0.f) {
          const FF nx = ff_add(run, x);
          if (!last && ff_gt(nx, tau)) {
            pick = j;
            tin = ff_add(tau, ff_neg(run));
            break;
          }
          pick = j;  // the last chunk with mass so far
          tin = x;
          run = nx;
        }
      }
      S.pick = pick;
      S.tau_in = tin;
    }
  }
  __syncthreads();
  const int jc = S.pick;
  if (jc < 0) return -1;  // no mass at all (flagged by the caller's checks)
  // ---- every thread: vector t of each 256-vector tile of the chunk, loaded
  // in batches of four per thread (each batch held in registers until it
  // lands); per-warp sums of r per tile --------------------------------------
  const int64_t e0 = static_cast<int64_t>(jc) * span, e1 = min(static_cast<int64_t>(V), e0 + span);
  const int nvc = static_cast<int>((e1 - e0 + VW - 1) / VW);
  const int ntile = (nvc + kThreads - 1) / kThreads;  // <= kDrawTiles (the caller checks)
  auto rfrom = [&](const typename E::Vec& v, int j, float (&r)[VW]) {
    float z[VW];
    E::unpack(v, z);
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const int64_t e = e0 + static_cast<int64_t>(j) * VW + k;
      const float p = ex2((z[k] - M) * c);
      r[k] = e == xex ? 0.f : (w.in(z[k], e) ? __fmul_rn(p, w.C) : p);
    }
  };
  auto rvals = [&](int j, float (&r)[VW]) { rfrom(load_vec<DT, VEC>(row, e0, e1, j), j, r); };
  constexpr int kBatch = 4;  // (8 spills registers elsewhere in the kernel)
  for (int h = 0; h < ntile; h += kBatch) {
    typename E::Vec raw[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int j = (h + q) * kThreads + t;
      if (h + q < ntile && j < nvc) raw[q] = load_vec<DT, VEC>(row, e0, e1, j);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = h + q, j = i * kThreads + t;
      float rsum = 0.f;
      if (i < ntile && j < nvc) {
        float r[VW];
        rfrom(raw[q], j, r);
#pragma unroll
        for (int k = 0; k < VW; ++k) rsum += r[k];
      }
      const float ws = warp_sum(rsum);
      if (lane == 0) S.tile[i][warp] = ws;
    }
  }
  __syncthreads();
  // ---- warp 0: lane i sums tile i; a float-float scan over tiles, then an
  // fp32 walk over the chosen tile's warps relative to the tile's start (the
  // same additions that formed the tile sum), locates the 32 vectors holding
  // U * R -----------------------------------------------------------------
  if (warp == 0) {
    const FF tin = S.tau_in;
    const bool fb = S.fallback != 0;
    float ti = 0.f;
    if (lane < ntile)
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) ti += S.tile[lane][w2];
    const FF incl = warp_ffscan(ff(ti), lane);
    const unsigned hit = fb ? 0u : __ballot_sync(0xffffffffu, ti > 0.f && ff_gt(incl, tin));
    const unsigned pos = __ballot_sync(0xffffffffu, ti > 0.f);
    const bool last = hit == 0;
    const int sel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == sel) {
      const float t = ff_add(tin, ff_neg(ff_add(incl, -ti))).hi;  // relative to the tile's start
      float run = 0.f, wb = 0.f;
      int ws = -1;
      for (int w2 = 0; w2 < kWarps; ++w2) {
        const float g = S.tile[lane][w2];
        const float nx = run + g;
        if (g > 0.f) {
          ws = w2;
          wb = run;
          if (!last && nx > t) break;
        }
        run = nx;
      }
      S.tsel = ws >= 0 ? lane : -1;
      S.wsel = ws;
      S.tw = t - wb;
      S.fallback = last ? 1 : 0;
    }
    if (lane == 0 && sel < 0) S.tsel = -1;
  }
  __syncthreads();
  const int ts = S.tsel;
  if (ts < 0) return -1;
  // ---- the chosen warp: a scan of its lanes' r sums in the chosen tile, then
  // the crossing lane walks its vector ---------------------------------------
  if (warp == S.wsel) {
    const int j = ts * kThreads + t;
    float r[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k) r[k] = 0.f;
    if (j < nvc) rvals(j, r);
    float vs = 0.f;
#pragma unroll
    for (int k = 0; k < VW; ++k) vs += r[k];
    const float tw = S.tw;  // relative to the warp's first vector of the tile
    const bool fb = S.fallback != 0;
    float inc = vs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const float exc = __shfl_up_sync(0xffffffffu, inc, 1);
    const unsigned hit = fb ? 0u : __ballot_sync(0xffffffffu, vs > 0.f && inc > tw);
    const unsigned pos = __ballot_sync(0xffffffffu, vs > 0.f);
    const bool lastel = hit == 0;  // past the end, or rounding inside the tile
    const int sel = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (lane == sel) {
      float run = lane > 0 ? exc : 0.f;
      int kk = -1, kl = -1;
#pragma unroll
      for (int k = 0; k < VW; ++k)
        if (r[k] > 0.f) {
          run += r[k];
          kl = k;
          if (!lastel && kk < 0 && run > tw) kk = k;
        }
      const int ksel = kk >= 0 ? kk : kl;  // rounding within the vector: its last r > 0
      float rt = 0.f;
#pragma unroll
      for (int k = 0; k < VW; ++k)
        if (k == ksel) rt = r[k];
      S.pick = ksel >= 0 ? static_cast<int>(e0 + static_cast<int64_t>(j) * VW + ksel) : -1;
      S.q = __fdiv_rn(rt, S.R.hi);
      S.fallback = (fb || kk < 0) ? 1 : 0;
    }
    if (lane == 0 && sel < 0) S.pick = -1;
  }
  __syncthreads();
  return S.pick;
}

// The final step of an inverse-CDF draw over a slice [v0, v1) of row n,
// run by one warp: the slice's per-warp segment sums segs[ntl * kWarps]
// (shared memory, tile-major) and the mass before the slice (pre) locate the
// segment where the running sum of r crosses tau, and a scan of its 32
// vectors the logit.  Lanes own contiguous blocks of segments; a float-float
// warp scan of the block sums finds the block that holds the crossing.
// Inside it the walk runs in fp32, relative to the block's start: tau less
// the mass before the block, rounded once, against the same additions that
// formed the block sum (so a crossing found by the scan is found again, and
// what rounding can move lies within a few ulps of the block's mass).
// last_pos: tau lies at or past the end (rounding), take the last logit with
// r > 0.  Returns the token in every lane (-1: no mass), and r at it in rv.
template <int DT, bool VEC>
__device__ __forceinline__ int owner_scan(const float* segs, int ntl, FF tau, FF pre, bool last_pos,
                                          const void* rowt, const void* rowd, int64_t v0,
                                          int64_t v1, int nv, int mode, float mt, float md, float c,
                                          float ist, float isd, int xn, const SgW& sgw, float& rv_out) {
  constexpr int VW = Elem<DT>::VW;
  const int lane = threadIdx.x & 31;
  const int nseg = ntl * kWarps;
  const int per = (nseg + 31) / 32;
  const int s0 = min(nseg, lane * per), s1 = min(nseg, s0 + per);
  float bsum = 0.f;
  int lastpos = -1;
  for (int sg = s0; sg < s1; ++sg) {
    const float g = segs[sg];
    if (g > 0.f) {
      bsum += g;
      lastpos = sg;
    }
  }
  const FF incl = warp_ffscan(ff(bsum), lane);
  const FF bpre = ff_add(pre, ff_add(incl, -bsum));
  const unsigned hitm = last_pos ? 0u
                                     : __ballot_sync(0xffffffffu, bsum > 0.f && ff_gt(ff_add(bpre, bsum), tau));
  const unsigned posm = __ballot_sync(0xffffffffu, lastpos >= 0);
  int seg = -1;
  float tseg = 0.f;  // U*R less the mass before the chosen segment
  if (hitm) {
    const int L = __ffs(hitm) - 1;
    if (lane == L) {
      const float t = ff_add(tau, ff_neg(bpre)).hi;
      float cum = 0.f;
      for (int sg = s0; sg < s1; ++sg) {
        const float g = segs[sg];
        if (g > 0.f) {
          const float nx = cum + g;
          if (nx > t) {
            seg = sg;
            tseg = t - cum;
            break;
          }
          cum = nx;
        }
      }
      if (seg < 0) seg = lastpos;  // rounding inside the block
    }
    seg = __shfl_sync(0xffffffffu, seg, L);
    tseg = __shfl_sync(0xffffffffu, tseg, L);
  }
  const int lastseg = posm ? __shfl_sync(0xffffffffu, lastpos, 31 - __clz(posm)) : -1;
  bool lp = last_pos || seg < 0;
  if (seg < 0) seg = lastseg;
  const int j = (seg / kWarps) * kThreads + (seg % kWarps) * 32 + lane;
  float r[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) r[k] = 0.f;
  if (seg >= 0 && j < nv)
    residual_vec<DT, VEC>(rowt, rowd, v0, v1, j, mode, mt, md, c, ist, isd, xn, sgw, r);
  const int32_t base = static_cast<int32_t>(v0) + j * VW;
  int found = -1;
  float rv = 0.f;  // r at the found logit (the sampler reports it as sigma(t))
  if (!lp) {
    // the segment's 32 vectors: an fp32 scan relative to the segment start
    float vs = 0.f;
#pragma unroll
    for (int k = 0; k < VW; ++k) vs += r[k];
    float inc = vs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const float exc = __shfl_up_sync(0xffffffffu, inc, 1);
    const unsigned m = __ballot_sync(0xffffffffu, vs > 0.f && inc > tseg);
    if (m) {
      if (lane == __ffs(m) - 1) {
        float run = lane > 0 ? exc : 0.f;
        int kk = -1, klast = -1;
#pragma unroll
        for (int k = 0; k < VW; ++k) {
          if (r[k] > 0.f) {
            run += r[k];
            klast = k;
            if (kk < 0 && run > tseg) kk = k;
          }
        }
        const int ksel = kk >= 0 ? kk : klast;
        found = base + ksel;
#pragma unroll
        for (int k = 0; k < VW; ++k)
          if (k == ksel) rv = r[k];
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
    if (m && lane == 31 - __clz(m)) {
      found = base + kl;
#pragma unroll
      for (int k = 0; k < VW; ++k)
        if (k == kl) rv = r[k];
    }
  }
  const unsigned mf = __ballot_sync(0xffffffffu, found >= 0);
  rv_out = mf ? __shfl_sync(0xffffffffu, rv, __ffs(mf) - 1) : 0.f;
  return mf ? __shfl_sync(0xffffffffu, found, __ffs(mf) - 1) : -1;
}

// What a batch row's decision needs besides the records, the same on every
// thread of every CTA that decides it.
struct RowCtx {
  int b;
  int kb_in;    // the row's drafts (an MSS node's candidates); -1: bad count
  int kb;       // max(kb_in, 0)
  int npos;     // positions with records: 0..npos
  int u_draw;   // the uniform of the final draw
  float T, c;   // temperature, log2(e)/T
  bool greedy, temp_ok, nd, sg_on;
  int64_t u0;   // first record unit and output row of the batch row
  RowLayout L;
};

template <int MODE>
__device__ __forceinline__ RowCtx row_ctx(const DecideParams& P, int b) {
  constexpr bool kTopF = MODE == kModeSsd;
  constexpr bool kSample = MODE == kModeSample;
  constexpr bool kMss = MODE == kModeMss;
  RowCtx X;
  X.b = b;
  X.T = P.temp[b];
  X.greedy = X.T == 0.f;
  X.temp_ok = X.T >= 0.f && X.T < pos_inf();
  X.c = X.greedy ? 1.f : temp_scale(X.T);
  // records, outputs: [B, K+1] (an MSS node has one position)
  X.u0 = kMss ? static_cast<int64_t>(b) : static_cast<int64_t>(b) * (P.K + 1);
  X.L = row_layout(P.cu, P.ntok, b, P.K, P.t_bs, P.t_rs, P.d_bs, P.d_rs);
  X.kb_in = X.L.kb;
  if (kMss && P.ncand) {
    const int m = P.ncand[b];
    X.kb_in = (m >= 0 && m <= P.K) ? m : -1;
  }
  X.kb = X.kb_in < 0 ? 0 : X.kb_in;
  X.npos = kMss ? 0 : X.kb;
  X.u_draw = kMss ? P.K : X.kb;
  X.nd = P.no_draft != 0;
  X.sg_on = (kSample || (kTopF && P.sg_F > 0)) && !X.greedy && X.temp_ok;
  return X;
}

// Shared memory of one batch row's decision.
struct PrepSmem {
  PosStats ps[kMaxK + 1];
  Dec dec;
  int32_t tok_slot;  // the token found by the final scan
  float q_slot;      // the sampler: sigma of that token
  float sg_d[kMaxK + 1];    // Saguaro: weighted mass of the top-F_s,
  float sg_zl[kMaxK + 1];   //   its F_s-th key (zl, il), and whether
  int32_t sg_il[kMaxK + 1]; //   the sent token is among them
  int32_t sg_xin[kMaxK + 1];
  float sg_kv[kMaxF];       // the sampler: its row's top-F_s keys
  int32_t sg_ki[kMaxF];
  int32_t sg_nk;
  int32_t copy_fail;        // a staged copy of the row's passes did not land in time
  int32_t pre_x[kMaxK];     // draft tokens, their logits and the uniforms,
  float pre_zt[kMaxK];      // fetched while the records are combined
  float pre_zd[kMaxK];
  float pre_u[kMaxK];
};

// The decision of batch row X.b from its chunk records, by every thread of
// one CTA: the records combined per position, the Saguaro keys of the draft
// rows, and the accept test (or the first MSS candidate's test), leaving the
// outcome in S.dec.  wkeys: key scratch of the first nkw warps (the others
// take no part in the key merges; nkw >= 1).  wait_primary: the
// records come from the previous kernel on the stream (wait for it once the
// inputs are fetched).  Ends with a CTA barrier.
template <int DT, int MODE>
__device__ __forceinline__ void decide_prepare(const DecideParams& P, const RowCtx& X, PrepSmem& S,
                                               WarpKeys* wkeys, int nkw, bool wait_primary) {
  using E = Elem<DT>;
  constexpr bool kSample = MODE == kModeSample;
  constexpr bool kMss = MODE == kModeMss;
  const int F = P.F;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const bool greedy = X.greedy, temp_ok = X.temp_ok, nd = X.nd, sg_on = X.sg_on;
  const float c = X.c;
  const int64_t u0 = X.u0;
  const RowLayout& L = X.L;
  const int kb_in = X.kb_in, kb = X.kb, npos = X.npos;
  // ---- every CTA combines the records and decides (identical results) -------
  // The last warp first fetches what the decision needs besides the records.
  if (warp == kWarps - 1) {
    for (int i = lane; i < kb; i += 32) {
      const int x = P.tokens[L.tok0 + i];
      float zt = 0.f, zd = 0.f;
      if (x >= 0 && x < P.V) {
        const int64_t ri = kMss ? 0 : i;  // every candidate of a node sits on its one row
        zt = E::scalar(static_cast<const char*>(P.zt) + (L.t_off + ri * P.t_rs) * E::ES, x);
        if (!nd) zd = E::scalar(static_cast<const char*>(P.zd) + (L.d_off + ri * P.d_rs) * E::ES, x);
      }
      S.pre_x[i] = x;
      S.pre_zt[i] = zt;
      S.pre_zd[i] = zd;
      S.pre_u[i] = P.unif[L.u_off + i];
    }
  }
  // Everything above reads only the call's inputs; the records below are
  // the row-statistics kernel's output, so wait for it to complete here.
  if (wait_primary) pdl_wait_primary();
  // Half a warp per position: positions 2w and 2w+1 on warp w, 16 per pass.
  for (int i0 = 2 * warp; i0 <= npos; i0 += 2 * kWarps) {
    const int i = i0 + (lane >> 4);
    const PosStats p = combine_position<16>(P.recs + (u0 + min(i, npos)) * P.nchunk, P.nchunk, c, lane & 15);
    if ((lane & 15) == 0 && i <= npos) S.ps[i] = p;
  }
  __syncthreads();

  // ---- Saguaro sampling ([SSD] §4.2.1): the drafts of an SSD round came from
  // sigma_{F_s,C}, and the sampler draws from it.  Per draft row: its top-F_s
  // keys (the lookahead's merged candidates, which exclude the sent token x,
  // with x put back in key order), their mass in units of 2^((z - Md) c), and
  // the F_s-th key.  One warp per row.  Greedy rows are left one-hot.
  if (sg_on) {
    const int nrows = kSample ? 1 : kb;
    const int ncand = static_cast<int>(P.nchunk) * F;
    const bool cta_rank = kSample && ncand <= kWarpCand;  // the sampler: all warps rank
    if (cta_rank) cta_rank_keys(P.cand_v + u0 * ncand, P.cand_i + u0 * ncand, ncand, F, wkeys[0]);
    for (int i = warp; warp < nkw && i < nrows; i += nkw) {
      const int64_t u = u0 + i;
      WarpTopF Lk;
      if (cta_rank) {
        Lk.init();
        if (lane < F) {
          Lk.v = wkeys[0].ov[lane];
          Lk.i = wkeys[0].oi[lane];
        }
      } else {
        Lk = warp_keys(P.cand_v + u * ncand, P.cand_i + u * ncand, ncand, F, lane, wkeys[warp]);
      }
      const int fs = P.sg_F;
      const int x = kSample ? -1 : S.pre_x[i];
      const float zx = kSample ? neg_inf() : S.pre_zd[i];
      const int pos = (x >= 0) ? __popc(__ballot_sync(0xffffffffu, lane < F && key_beats(Lk.v, Lk.i, zx, x)))
                               : F;
      const bool xin = x >= 0 && pos < fs;
      const int fl = xin ? fs - 1 : fs;  // list entries inside the top-F_s
      const float Md = S.ps[i].Md;
      float d = (lane < fl && Lk.i != INT_MAX) ? ex2((Lk.v - Md) * c) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (xin) d += ex2((zx - Md) * c);
      // the F_s-th key of the list with x inserted at pos
      const int src = (!xin) ? fs - 1 : (pos == fs - 1 ? -1 : fs - 2);
      const float lv = __shfl_sync(0xffffffffu, Lk.v, src < 0 ? 0 : src);
      const int32_t li = __shfl_sync(0xffffffffu, Lk.i, src < 0 ? 0 : src);
      if (lane == 0) {
        S.sg_d[i] = d;
        S.sg_zl[i] = src < 0 ? zx : lv;
        S.sg_il[i] = src < 0 ? x : li;
        S.sg_xin[i] = xin;
      }
      if (kSample) {  // the keys themselves, for the chunk-local draw
        const bool valid = lane < fs && Lk.i != INT_MAX;
        if (valid) {
          S.sg_kv[lane] = Lk.v;
          S.sg_ki[lane] = Lk.i;
        }
        const unsigned vm = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) S.sg_nk = __popc(vm);
      }
    }
    __syncthreads();
  }
  // ---- MSS at a token-tree node ([CS349D] §6.4): warp 0 tests the first
  // candidate; each rejection is followed by a residual pass below ------------
  if (kMss && warp == 0) {
    const PosStats& q = S.ps[0];
    int nf = 0;
    if (lane == 0 && temp_ok)
      nf = greedy ? ((q.bad & 1) || q.it == INT_MAX || q.id == INT_MAX)
                  : (!(q.St.hi >= 1.f) || q.Mt == kNegMax || !(q.Sd.hi >= 1.f) || q.Md == kNegMax);
    const bool cl = lane < kb;
    const int x = cl ? S.pre_x[lane] : -1;
    int status = temp_ok ? 0 : kBadTemp;
    if (kb_in < 0) status |= kBadCount;
    if (__any_sync(0xffffffffu, nf)) status |= kNonFinite;
    if (q.bad & 2) status |= kTimeout;
    if (__any_sync(0xffffffffu, cl && (x < 0 || x >= P.V))) status |= kBadToken;
    const bool ok = !(status & kErrors);
    const bool naive = P.naive != 0;
    // t_j = p(x_j) / q(x_j), from the log2 difference so neither factor
    // underflows; q(x_j) > 0 iff its draft logit is finite
    float t = 0.f;
    bool qpos = false;
    if (cl && ok && !greedy) {
      const float lt = __fmul_rn(S.pre_zt[lane] - q.Mt, c);
      const float ld = __fmul_rn(S.pre_zd[lane] - q.Md, c);
      qpos = S.pre_zd[lane] != neg_inf();
      t = qpos ? __fmul_rn(ex2(__fsub_rn(lt, ld)), __fdiv_rn(q.Sd.hi, q.St.hi)) : 0.f;
    }
    const unsigned hitg = __ballot_sync(0xffffffffu, ok && cl && greedy && x == q.it);
    const int acc_g = hitg ? __ffs(hitg) - 1 : -1;
    const bool a0 = __shfl_sync(0xffffffffu, cl && qpos && t >= S.pre_u[lane < kMaxK ? lane : 0], 0);
    float ap = 0.f;
    if (ok && cl && !naive) ap = greedy ? (lane == acc_g ? 1.f : 0.f) : (lane == 0 ? fminf(t, 1.f) : 0.f);
    S.dec.ap[lane] = ap;
    S.dec.px[lane] = t;
    S.dec.qx[lane] = qpos ? 1.f : 0.f;
    if (lane == 0) {
      int acc = -1, token = -1, mode = 1, need = 0;
      if (ok) {
        if (greedy) {
          acc = acc_g;
          token = q.it;
        } else if (naive || kb == 0) {
          need = 1;  // a draw from p itself
        } else if (a0) {
          acc = 0;
          token = S.pre_x[0];
        } else {
          need = 1;  // residual max(0, p - c_1 q), c_1 = 1
          mode = 0;
        }
      }
      S.dec.n = 0;
      S.dec.status = status;
      S.dec.mode = mode;
      S.dec.xn = -1;
      S.dec.need_scan = need;
      S.dec.token = token;
      S.dec.acc = acc;
      S.dec.owner = -1;
      S.dec.last_pos = 0;
      S.dec.mt = q.Mt;
      S.dec.md = q.Md;
      S.dec.ist = __fdiv_rn(1.f, q.St.hi);
      S.dec.isd = __fdiv_rn(1.f, q.Sd.hi);
      S.dec.sgc = 1.f;
      S.dec.zl = pos_inf();
      S.dec.il = -1;
      S.dec.full_pass = 0;
      S.dec.tau = ff(0.f);
      S.dec.pre_mine = ff(0.f);
      S.dec.R = ff(0.f);
      S.dec.cff = ff(1.f);
      S.dec.cq = 1.f;
      S.dec.next = 1;
      S.dec.again = 0;
      S.tok_slot = token;
      S.q_slot = 0.f;
      S.copy_fail = 0;
    }
  }
  if (!kMss && warp == 0) {
    int nf = 0;
    // Saguaro: the weighted normaliser of draft row i, sum - (1 - C) * top-F_s mass
    const float sgC = sg_on ? P.sg_C : 1.f;
    const FF one_m_c = two_sum(1.f, -sgC);  // 1 - C, exactly
    auto sdp = [&](int i) -> FF {
      return sg_on ? ff_add(S.ps[i].Sd, ff_neg(ff_mul(one_m_c, S.sg_d[i]))) : S.ps[i].Sd;
    };
    if (kSample && temp_ok && lane == 0) {  // the sampled row sits in the draft fields
      const PosStats& q = S.ps[0];
      nf = greedy ? ((q.bad & 1) || q.id == INT_MAX)
                  : (!(q.Sd.hi >= 1.f) || q.Md == kNegMax || !(sdp(0).hi > 0.f));
    } else if (!kSample && lane <= kb && temp_ok) {
      const PosStats& q = S.ps[lane];
      const bool d_full = lane < kb && !nd;  // draft rows that are normalised
      const bool d_any = (MODE != kModeVerify) || d_full;
      if (greedy) {
        nf = (q.bad & 1) || q.it == INT_MAX || (d_full && q.id == INT_MAX);
      } else {
        nf = !(q.St.hi >= 1.f) || q.Mt == kNegMax;
        if (d_full) nf |= !(q.Sd.hi >= 1.f) || q.Md == kNegMax || !(sdp(lane).hi > 0.f);
        else if (d_any) nf |= q.Sd.hi != q.Sd.hi;  // draft row K: NaN / +inf only
      }
    }
    const bool acc_lane = lane < kb;
    const int x = acc_lane ? S.pre_x[lane] : -1;
    int status = temp_ok ? 0 : kBadTemp;
    if (kb_in < 0) status |= kBadCount;
    if (__any_sync(0xffffffffu, nf)) status |= kNonFinite;
    if (__any_sync(0xffffffffu, lane <= kb && (S.ps[lane].bad & 2))) status |= kTimeout;
    if (__any_sync(0xffffffffu, acc_lane && (x < 0 || x >= P.V))) status |= kBadToken;
    const bool ok = !(status & kErrors);
    bool accept = false;
    float px = 0.f, qx = 0.f;
    if (acc_lane && ok) {
      const PosStats& q = S.ps[lane];
      if (greedy) {  // one-hot p and q (q at x itself without draft logits)
        px = (x == q.it) ? 1.f : 0.f;
        qx = (nd || x == q.id) ? 1.f : 0.f;
        accept = (x == q.it) && (nd || x == q.id);
      } else if (nd) {  // q_i(x_i) = 1: accept iff p_i(x_i) >= u
        const float lt = __fmul_rn(S.pre_zt[lane] - q.Mt, c);
        px = __fdiv_rn(ex2(lt), q.St.hi);
        qx = 1.f;
        accept = px >= S.pre_u[lane];
      } else {
        const float ztx = S.pre_zt[lane];
        const float zdx = S.pre_zd[lane];
        const float lt = __fmul_rn(ztx - q.Mt, c);  // log2 of unnormalised p_i(x), q_i(x)
        const float ld = __fmul_rn(zdx - q.Md, c);
        const float St = q.St.hi, Sd = sdp(lane).hi;
        const float wx = (sg_on && S.sg_xin[lane]) ? sgC : 1.f;  // Saguaro weight of x_i
        px = __fdiv_rn(ex2(lt), St);
        qx = __fdiv_rn(__fmul_rn(ex2(ld), wx), Sd);
        if (zdx != neg_inf() && wx > 0.f) {  // q_i(x_i) > 0
          const float ratio = __fdiv_rn(__fmul_rn(ex2(__fsub_rn(lt, ld)), __fdiv_rn(Sd, St)), wx);
          accept = ratio >= S.pre_u[lane];
        }
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, acc_lane && !accept);
    const int n = ok ? (rej ? __ffs(rej) - 1 : kb) : 0;
    if (lane < kb) {
      S.dec.px[lane] = px;
      S.dec.qx[lane] = qx;
    }
    if (lane == 0) {
      const PosStats& q = S.ps[n];
      S.dec.n = n;
      S.dec.status = status;
      S.dec.mode = kSample ? 3 : (n < kb) ? (nd ? 2 : 0) : 1;
      S.dec.xn = (n < kb) ? S.pre_x[n] : -1;
      S.dec.need_scan = ok && !greedy;
      S.dec.token = (ok && greedy) ? (kSample ? q.id : q.it) : -1;
      S.dec.owner = -1;
      S.dec.last_pos = 0;
      // the sampler's row statistics are the draft fields of position 0
      S.dec.mt = kSample ? q.Md : q.Mt;
      S.dec.md = q.Md;
      S.dec.ist = __fdiv_rn(1.f, (kSample ? sdp(0) : q.St).hi);
      S.dec.isd = __fdiv_rn(1.f, ((n < kb) ? sdp(n) : q.Sd).hi);
      // Saguaro weights on the residual: the draft row n (mode 0) or the row (mode 3)
      const bool weighted = sg_on && (kSample || (n < kb && !nd));
      S.dec.sgc = weighted ? sgC : 1.f;
      S.dec.zl = weighted ? S.sg_zl[n] : pos_inf();
      S.dec.il = weighted ? S.sg_il[n] : -1;
      // The chunk-local draw takes the weighted mass from the chunk sums less
      // (1 - C) x the keys' mass; when that correction is most of the row's
      // mass the difference loses fp32 precision, and the draw reads the whole
      // row instead (its residual total is then summed from the weighted
      // values themselves).
      S.dec.full_pass = (kSample && sg_on) ? (__fmul_rn(one_m_c.hi, S.sg_d[0]) > 0.5f * q.Sd.hi) : 0;
      // Without draft probabilities the residual at a rejection is p_n less
      // its rejected token: the same draw with that token's mass taken from
      // its chunk, or the whole row when the token holds most of the mass.
      S.dec.zx = (n < kb && nd) ? S.pre_zt[n] : 0.f;
      if (!kSample && n < kb && nd)
        S.dec.full_pass = ex2(__fmul_rn(S.dec.zx - q.Mt, c)) > 0.5f * q.St.hi;
      S.dec.tau = ff(0.f);
      S.dec.pre_mine = ff(0.f);
      S.tok_slot = S.dec.token;
      S.q_slot = (ok && greedy) ? 1.f : 0.f;
      S.copy_fail = 0;
    }
  }
  __syncthreads();

}

template <int DT, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads, 4) decide_kernel(const DecideParams P) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  constexpr bool kTopF = MODE == kModeSsd;      // outcome keys and hit
  constexpr bool kSample = MODE == kModeSample;  // draft-side Saguaro sampling
  constexpr bool kMss = MODE == kModeMss;        // candidates at token-tree nodes
  extern __shared__ float segs[];  // [tiles * kWarps] segment sums of r
  __shared__ PrepSmem S;
  __shared__ FF cta_total[2];  // this CTA's residual mass, per attempt
  __shared__ DrawSmem draw;
  __shared__ RingBars ring_bars;
  __shared__ WarpKeys wkeys[(kTopF || kSample) ? kWarps : 1];

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CB = P.CB;
  const int b = static_cast<int>(blockIdx.x / CB);
  const int K = P.K, F = P.F;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const RowCtx X = row_ctx<MODE>(P, b);
  const float c = X.c;
  const int64_t u0 = X.u0;
  const RowLayout& L = X.L;
  const int kb = X.kb, u_draw = X.u_draw;
  const bool sg_on = X.sg_on;
  decide_prepare<DT, MODE>(P, X, S, wkeys, (kTopF || kSample) ? kWarps : 1, true);

  // ---- a draw from a whole row's own distribution (the bonus after K accepted
  // drafts, the sampler) needs only the one chunk holding U * R: rank 0 finds
  // it from the chunk records and reads that chunk alone -----------------------
  // (P.local_draw: the host's choice, made when a chunk is shorter than one
  // CTA's slice of the row and holds at most kDrawTiles tiles)
  const bool local_draw = S.dec.need_scan && P.local_draw &&
                          (S.dec.mode == 1 || ((S.dec.mode == 3 || S.dec.mode == 2) && !S.dec.full_pass));
  const bool scan = S.dec.need_scan && !local_draw;  // the residual pass over row n
  if (local_draw && rank == 0) {
    const int nn = S.dec.n;
    const char* row = kSample ? static_cast<const char*>(P.zd) + L.d_off * E::ES
                              : static_cast<const char*>(P.zt) +
                                    (L.t_off + static_cast<int64_t>(nn) * P.t_rs) * E::ES;
    const SgW w = kSample ? SgW{S.dec.sgc, S.dec.zl, S.dec.il} : SgW{1.f, pos_inf(), -1};
    const int tok = chunk_draw<DT, VEC>(P.recs + (u0 + nn) * P.nchunk, P.nchunk, P.chunk, P.V,
                                        kSample, S.dec.mt, c, row,
                                        P.unif[L.u_off + u_draw], S.sg_kv, S.sg_ki,
                                        (kSample && sg_on) ? S.sg_nk : 0, w, kSample ? P.pieces : 0,
                                        (kSample && P.pieces) ? P.piece_stats + (u0 + nn) * P.nchunk * kMaxPieces
                                                              : nullptr,
                                        S.dec.mode == 2 ? S.dec.xn : -1, S.dec.zx, draw);
    if (threadIdx.x == 0) {
      S.tok_slot = tok;
      S.q_slot = draw.q;
      if (draw.fallback) S.dec.status |= kFallback;
    }
    __syncthreads();
  }

  // ---- this CTA's slice of row n; aligned rows start streaming it now, so the
  // copies run while the keys are merged ------------------------------------
  const int n_dec = S.dec.n;
  Chunk RC;
  RC.b = b;
  RC.i = n_dec;
  RC.rowt = kSample  // the sampler reads its one row through the target slot
                ? static_cast<const char*>(P.zd) + L.d_off * E::ES
                : static_cast<const char*>(P.zt) + (L.t_off + static_cast<int64_t>(n_dec) * P.t_rs) * E::ES;
  RC.rowd = (S.dec.mode == 0)  // draft row n, read only for the residual max(p - q, 0)
                ? static_cast<const char*>(P.zd) + (L.d_off + static_cast<int64_t>(n_dec) * P.d_rs) * E::ES
                : nullptr;
  RC.v0 = static_cast<int64_t>(rank) * P.L;
  RC.v1 = min(static_cast<int64_t>(P.V), RC.v0 + P.L);
  RC.nv = RC.v1 > RC.v0 ? static_cast<int>((RC.v1 - RC.v0 + VW - 1) / VW) : 0;
  unsigned char* ring = reinterpret_cast<unsigned char*>(segs) + P.ring_off;
  const bool staged = VEC && scan && P.stages > 0;
  if (staged) {
    Chunk SC = RC;
    if (S.dec.mode != 0) SC.rowd = nullptr;  // mode 1 reads p_n only
    ring_start<DT>(ring_bars, ring, P.stages, SC, P.stall == b + 1 && rank == 0, !kMss);
    __syncthreads();
  }

  if (scan) {
    const SgW sgw{S.dec.sgc, S.dec.zl, S.dec.il};
    const void* rowt = RC.rowt;
    const void* rowd = RC.rowd;
    const int64_t v0 = RC.v0;
    const int64_t v1 = RC.v1;
    const int nv = RC.nv;
    const int ntl = (nv + kThreads - 1) / kThreads;
    bool copies_ok = true;
    // ---- residual mass of this slice: per-warp segment sums.  One pass, plus
    // one when a zero mass falls back to p; an MSS node one per rejection ----
    const int max_pass = kMss ? kb + 2 : 2;
    for (int pass = 0; pass < max_pass; ++pass) {
      const int mode = S.dec.mode;
      const float mt = S.dec.mt, md = S.dec.md, ist = S.dec.ist;
      const float isd = kMss ? __fmul_rn(S.dec.isd, S.dec.cq) : S.dec.isd;  // MSS: c_j q
      // (a CTA whose copies gave up reads its later passes directly: its ring
      // may still have a copy in flight, and the row is an error row anyway)
      if (staged && (pass == 0 || copies_ok)) {
        Chunk SC = RC;
        if (mode != 0) SC.rowd = nullptr;
        if (pass > 0) {  // another pass over the slice (an MSS rejection, a fallback)
          __syncthreads();
          ring_reset(ring_bars, P.stages);
          ring_start<DT>(ring_bars, ring, P.stages, SC, false, !kMss);
          __syncthreads();
        }
        copies_ok = ring_residual<DT>(ring_bars, ring, P.stages, SC, mode, mt, md, c, ist, isd,
                                      S.dec.xn, sgw, segs, ntl, !kMss) && copies_ok;
      } else
      for (int t0 = 0; t0 < ntl; t0 += kTileUnroll) {
        float s[kTileUnroll];
#pragma unroll
        for (int q = 0; q < kTileUnroll; ++q) {
          const int j = (t0 + q) * kThreads + threadIdx.x;
          s[q] = 0.f;
          if (j < nv) {
            float r[VW];
            residual_vec<DT, VEC>(rowt, rowd, v0, v1, j, mode, mt, md, c, ist, isd, S.dec.xn, sgw, r);
#pragma unroll
            for (int k = 0; k < VW; ++k) s[q] += r[k];
          }
        }
#pragma unroll
        for (int q = 0; q < kTileUnroll; ++q) {
          const float w = warp_sum(s[q]);
          if (lane == 0 && t0 + q < ntl) segs[(t0 + q) * kWarps + warp] = w;
        }
      }
      __syncthreads();
      if (warp == 0) {
        FF acc = ff(0.f);
        for (int sg = lane; sg < ntl * kWarps; sg += 32) acc = ff_add(acc, segs[sg]);
        acc = warp_ffsum_all(acc);
        if (lane == 0) cta_total[pass & 1] = acc;
      }
      cluster_sync();  // (1) per-CTA totals visible; every CTA of the cluster has started
      if (!copies_ok && threadIdx.x == 0) *cluster.map_shared_rank(&S.copy_fail, 0) = 1;
      if (warp == 0) {
        const FF tr = (lane < CB) ? *cluster.map_shared_rank(&cta_total[pass & 1], lane) : ff(0.f);
        const FF incl = warp_ffscan(tr, lane);
        const FF R = shfl(incl, 31);
        const FF tau = ff_mul(R, P.unif[L.u_off + u_draw]);  // the bonus uniform
        const unsigned own = __ballot_sync(0xffffffffu, tr.hi > 0.f && ff_gt(incl, tau));
        const unsigned pos = __ballot_sync(0xffffffffu, tr.hi > 0.f);
        const FF pm = shfl(ff_add(incl, ff_neg(tr)), rank);
        if (lane == 0) {
          S.dec.tau = tau;
          S.dec.pre_mine = pm;
          S.dec.R = R;
          S.dec.again = 0;
          if (kMss && mode == 0 && S.dec.next < kb && R.hi > 0.f) {
            // MSS: R = D_j; candidate j is accepted iff
            // p_j(x_j)/q(x_j) = max(0, t_j - c_j) / D_j >= u_j
            const int j = S.dec.next;
            const FF d = ff_add(ff(S.dec.px[j]), ff_neg(S.dec.cff));
            const float a = (S.dec.qx[j] > 0.f && d.hi > 0.f) ? __fdiv_rn(d.hi, R.hi) : 0.f;
            S.dec.ap[j] = fminf(a, 1.f);
            if (S.dec.qx[j] > 0.f && a >= S.pre_u[j]) {
              S.dec.acc = j;
              S.dec.token = S.pre_x[j];
              S.tok_slot = S.pre_x[j];
            } else {  // rejected: c_{j+1} = c_j + D_j, one more pass
              S.dec.cff = ff_add(S.dec.cff, R);
              S.dec.cq = S.dec.cff.hi;
              S.dec.next = j + 1;
              S.dec.again = 1;
            }
          } else if (R.hi > 0.f) {
            if (own) {
              S.dec.owner = __ffs(own) - 1;
            } else {  // U*R >= R after rounding: the last index with r > 0
              S.dec.owner = 31 - __clz(pos);
              S.dec.last_pos = 1;
              S.dec.status |= kFallback;
            }
          } else if (S.dec.mode != 1) {
            S.dec.mode = 1;  // zero residual mass: draw from p_n instead
            S.dec.status |= kFallback;
            S.dec.again = 1;
          }
        }
      }
      __syncthreads();  // the decision on the owner, made by warp 0, seen by the CTA
      if (!S.dec.again) break;
    }

    // ---- owner CTA: locate the crossing segment, then scan it --------------
    if (rank == S.dec.owner && warp == 0) {
      float rq;
      const int tok = owner_scan<DT, VEC>(segs, ntl, S.dec.tau, S.dec.pre_mine, S.dec.last_pos != 0,
                                          rowt, rowd, v0, v1, nv, S.dec.mode, S.dec.mt, S.dec.md, c,
                                          S.dec.ist, kMss ? __fmul_rn(S.dec.isd, S.dec.cq) : S.dec.isd,
                                          S.dec.xn, sgw, rq);
      if (lane == 0) {
        *cluster.map_shared_rank(&S.tok_slot, 0) = tok;
        // sigma(t) = r(t) / R: the pass's own total, free of the cancellation
        // in the weighted normaliser
        if (kSample) *cluster.map_shared_rank(&S.q_slot, 0) = __fdiv_rn(rq, S.dec.R.hi);
      }
    }
  }
  // ---- outcome keys, while the owner CTA's warp 0 scans: warps 1..7 of CTA
  // r merge lookaheads r, r + CB, ... (one warp each, all at once) -----------
  if (kTopF && warp > 0) {
    const bool ok = !(S.dec.status & kErrors);
    for (int k = rank + (warp - 1) * CB; k <= K; k += CB * (kWarps - 1)) {
      const int64_t u = u0 + k;
      const WarpTopF L = warp_keys(P.cand_v + u * P.nchunk * F, P.cand_i + u * P.nchunk * F,
                                   static_cast<int>(P.nchunk) * F, F, lane, wkeys[warp], P.fk[k]);
      if (lane < F) {
        const bool good = ok && lane < P.fk[k] && L.i != INT_MAX;
        P.keys[u * F + lane] = good ? L.i : -1;
        if (P.key_logits) P.key_logits[u * F + lane] = good ? L.v : neg_inf();
      }
    }
  }
  // The barrier's release/acquire ordering (cluster scope) makes the owner's
  // token (written into rank 0's shared memory after the first cluster
  // barrier) and every CTA's key writes (global memory) visible to rank 0; no
  // CTA exits while another may still read its shared memory.  Every CTA
  // passes here exactly once when a scan or keys ran.
  if (scan || kTopF) cluster_sync();

  // ---- outputs, written by rank 0 ---------------------------------------------
  if (kMss && rank == 0) {  // a node: its token, the accepted candidate, accept probabilities
    const int status = S.dec.status | (S.copy_fail ? kTimeout : 0);
    const bool ok = !(status & kErrors);
    const int t = threadIdx.x;
    const int32_t token = ok ? S.tok_slot : -1;
    if (t == 0) {
      int acc = ok ? S.dec.acc : -1;
      if (ok && P.naive) {  // naive sampling: the first candidate equal to the draw
        acc = -1;
        for (int j = 0; j < kb; ++j)
          if (S.pre_x[j] == token) {
            acc = j;
            break;
          }
      }
      P.out_tokens[b] = token;
      P.mss_acc[b] = acc;
      if (P.row_status) P.row_status[b] = ok ? (status & kFallback) : (status & kErrors);
    }
    if (P.mss_ap && t < K) P.mss_ap[static_cast<int64_t>(b) * K + t] = (ok && t < kb) ? S.dec.ap[t] : 0.f;
  }
  if (!kMss && rank == 0) {
    // A slice whose staged copies did not land makes the row an error row
    // (read after the barrier above, so the same on every thread).
    const int status = S.dec.status | (S.copy_fail ? kTimeout : 0);
    const bool ok = !(status & kErrors);
    const int n = S.dec.n;
    const int t = threadIdx.x;
    const int32_t token = S.tok_slot;
    if (t <= K) {
      int32_t v = -1;
      if (ok) v = (t < n) ? S.pre_x[t] : (t == n ? token : -1);
      P.out_tokens[u0 + t] = v;
    }
    if (t < K) {
      if (t < kb && P.p_draft) P.p_draft[L.tok0 + t] = ok ? S.dec.px[t] : 0.f;
      if (t < kb && P.q_draft) P.q_draft[L.tok0 + t] = ok ? S.dec.qx[t] : 0.f;
    }
    if (kTopF && S.copy_fail)
      for (int e = t; e < (K + 1) * F; e += kThreads) {
        P.keys[u0 * F + e] = -1;
        if (P.key_logits) P.key_logits[u0 * F + e] = neg_inf();
      }
    if (t == 0) {
      if (kSample) {
        if (P.q_draft) P.q_draft[b] = ok ? S.q_slot : 0.f;  // sigma(token)
      } else {
        P.accept_len[b] = ok ? n : 0;
      }
      if (P.row_status) P.row_status[b] = ok ? (status & kFallback) : (status & kErrors);
      if (P.hit) {
        uint8_t h = 0;
        if (ok && token >= 0)
          for (int f = 0; f < F; ++f) h |= (P.keys[(u0 + n) * F + f] == token);
        P.hit[b] = h;
      }
    }
  }
}

// Outcome keys alone (specv_predict_outcomes): one CTA per batch row, one warp
// per lookahead.  A lookahead whose sent token is out of range or whose draft
// row holds NaN / +inf gets -1 keys; the batch row's status ORs them.
struct PredictKeysParams {
  const int32_t* tokens;
  const ChunkRec* recs;
  const float* cand_v;
  const int32_t* cand_i;
  int32_t* keys;
  float* key_logits;
  int32_t* row_status;
  int32_t B, K, V, F, nchunk;
  int32_t fk[kMaxK + 1];  // keys kept at lookahead k
};

}  // namespace specv
