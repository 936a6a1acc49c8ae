// The Saguaro sampler's decision with one warp per row ("Speculative
// Speculative Decoding" §4.2.1: sigma_{F,C} puts weight C on the row's top-F
// logits and 1 elsewhere, renormalised; the draft token is drawn from it by
// inverse CDF of U, §2.1).
//
// The row-statistics kernel has already read every row once and left, per
// chunk, its record (the chunk's max and sum of 2^((z - max) c)), the same
// for each of its pieces (eighths of 32-trip chunks) and its top-F
// candidates.  A row's draw then needs only the piece that holds U * R.  One
// warp per row does every step of it:
//   1. combine the row's chunk records (one lane per chunk),
//   2. merge the chunks' candidate lists into the row's top-F_s keys,
//   3. the weighted mass R = S - (1 - C) x (the keys' mass) and the checks,
//   4. a float-float scan over the pieces' masses (the key corrections
//      subtracted from the pieces that hold them) finds the piece holding U*R,
//   5. that piece is read in batches of 16 warp tiles (32 16-byte vectors
//      each, coalesced) and summed unweighted in paired fp32 steps; a
//      butterfly leaves one tile's sum in each lane, the keys' weights are
//      applied per tile, a float-float scan over the tiles finds the tile, an
//      fp32 scan over its lanes (weighted values, recomputed) the vector, and
//      the crossing lane walks its elements.
// All rows of a launch are in flight at once (8 per CTA, two CTAs per SM), so
// the pieces stream at HBM rate, where one CTA per row left most of its
// warps waiting at barriers.
//
// Rows whose keys hold so much of the mass that the pieces' masses lose
// fp32 precision to the correction (the same test as the CTA-per-row kernel)
// are left to a CTA-wide pass over the whole row at the end of the CTA: its
// eight warps sum the row's weighted values tile by tile, and warp 0 locates
// the logit (the same pass and scan as the CTA-per-row kernel with one CTA
// per row).
#pragma once

#include "decide_kernel.cuh"

namespace specv {

constexpr int kSampleBatch = 16;  // warp tiles loaded per batch (16 x 16 B per lane)

struct PendRow {  // a row left for the CTA-wide pass, as its warp decided it
  const char* row;
  float mt, c, ist, U;
  SgW w;
  int32_t status;
  int32_t b;
  int64_t u0;  // its output slot
};

// Steps 4-5 for one row by one warp.  piece_stats: the row's piece table; row: the
// row's logits; M, c: its max and log2(e)/T; U: its uniform; keys: its top-F_s
// keys (value, index) in the warp's shared scratch, nk of them; w: the
// weights.  Returns the token in every lane (-1: no mass), with r(t) / R in
// q and `fb` set when rounding left U * R at or past the end of what was
// located (the last logit with r > 0 is then taken).
template <int DT>
__device__ __forceinline__ int warp_piece_draw(const float2* piece_stats, int nchunk, int32_t chunk, int pieces, int V,
                                              float M, float c, const char* row, float U,
                                              const float* kv, const int32_t* ki, int nk,
                                              const SgW& w, float& q, bool& fb) {
  using E = Elem<DT>;
  using Vec = typename E::Vec;
  constexpr int VW = E::VW;
  const int lane = threadIdx.x & 31;
  const int nloc = pieces * nchunk;
  const int32_t span = chunk / pieces;  // logits per piece
  const FF one_m_c = two_sum(1.f, -w.C);
  // ---- step 4: lanes over contiguous runs of pieces ---------------------------
  const int per = (nloc + 31) / 32;
  const int j0 = min(nloc, lane * per), j1 = min(nloc, j0 + per);
  auto mass = [&](int j) -> FF {  // piece j % pieces of chunk j / pieces
    FF x = piece_mass(piece_stats + static_cast<int64_t>(j / pieces) * kMaxPieces, j % pieces, M, c);
    for (int k = 0; k < nk; ++k)  // the weighted keys of this piece
      if (ki[k] / span == j) x = ff_add(x, ff_neg(ff_mul(one_m_c, ex2((kv[k] - M) * c))));
    return x.hi > 0.f ? x : ff(0.f);
  };
  FF mine = ff(0.f);
  for (int j = j0; j < j1; ++j) mine = ff_add(mine, mass(j));
  const FF incl = warp_ffscan(mine, lane);
  const FF R = shfl(incl, 31);
  const FF tau = ff_mul(R, U);
  const unsigned hit = __ballot_sync(0xffffffffu, mine.hi > 0.f && ff_gt(incl, tau));
  const unsigned pos = __ballot_sync(0xffffffffu, mine.hi > 0.f);
  bool last = hit == 0;  // U * R at or past the end after rounding
  const int owner = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  q = 0.f;
  fb = last;
  if (owner < 0) return -1;  // no mass at all (the caller's checks flag such rows)
  int pick = -1;
  FF tin = ff(0.f);  // U * R less the mass before the chosen piece
  if (lane == owner) {
    FF run = ff_add(incl, ff_neg(mine));
    for (int j = j0; j < j1; ++j) {
      const FF x = mass(j);
      if (x.hi > 0.f) {
        const FF nx = ff_add(run, x);
        if (!last && ff_gt(nx, tau)) {
          pick = j;
          tin = ff_add(tau, ff_neg(run));
          break;
        }
        pick = j;  // the last piece with mass so far
        tin = x;
        run = nx;
      }
    }
  }
  pick = __shfl_sync(0xffffffffu, pick, owner);
  tin = shfl(tin, owner);

  // ---- step 5: the chosen piece, tile by tile ---------------------------------
  const int64_t e0 = static_cast<int64_t>(pick) * span;
  const int64_t e1 = min(static_cast<int64_t>(V), e0 + span);
  const int nvc = static_cast<int>((e1 - e0 + VW - 1) / VW);
  const int ntile = (nvc + 31) / 32;
  // The keys inside this piece: lane k < nk holds key k's tile and (1 - C) x
  // its mass, subtracted from that tile's sum of 2^((z - M) c) below (the
  // loop sums every logit unweighted: identical to summing the weighted
  // values, up to rounding, since the keys are exactly the logits C weighs).
  int ktile = -1;
  float kcorr = 0.f;
  if (lane < nk) {
    const int64_t ix = ki[lane];
    if (ix >= e0 && ix < e1) {
      ktile = static_cast<int>((ix - e0) / (32 * VW));
      kcorr = __fmul_rn(one_m_c.hi, ex2((kv[lane] - M) * c));
    }
  }
  const unsigned kmask = __ballot_sync(0xffffffffu, ktile >= 0);
  const uint64_t mm = f2(M, M), cc = f2(c, c);
  auto rvals = [&](const Vec& v, int j, float (&r)[VW]) {
    float z[VW];
    E::unpack(v, z);
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      const float p = ex2((z[k] - M) * c);
      r[k] = w.in(z[k], e0 + static_cast<int64_t>(j) * VW + k) ? __fmul_rn(p, w.C) : p;
    }
  };
  FF run = ff(0.f);  // mass of the tiles before the current batch
  int tsel = -1, tlast = -1;
  float tw = 0.f, twlast = 0.f;  // U * R less the mass before the chosen (last positive) tile
  for (int t0 = 0; t0 < ntile && tsel < 0; t0 += kSampleBatch) {
    Vec raw[kSampleBatch];
#pragma unroll
    for (int g = 0; g < kSampleBatch; ++g) {
      const int j = (t0 + g) * 32 + lane;
      if (j < nvc) raw[g] = load_vec<DT, true>(row, e0, e1, j);
    }
    float a[kSampleBatch];
#pragma unroll
    for (int g = 0; g < kSampleBatch; ++g) {  // paired fp32 steps, two logits each
      const int j = (t0 + g) * 32 + lane;
      a[g] = 0.f;
      if (j < nvc) {
        float z[VW];
        E::unpack(raw[g], z);
        uint64_t acc = f2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VW; k += 2) {
          float x0, x1;
          f2_split(f2_mul(f2_sub(f2(z[k], z[k + 1]), mm), cc), x0, x1);
          acc = f2_add(acc, f2(ex2(x0), ex2(x1)));
        }
        float lo, hi;
        f2_split(acc, lo, hi);
        a[g] = lo + hi;
      }
    }
    // butterfly: after the stage of offset o each lane keeps the half of its
    // values selected by bit o of its lane and adds its partner's; lane l ends
    // with tile t0 + (l & 15) summed over the 16 lanes sharing bit 4, then
    // over both halves of the warp
#pragma unroll
    for (int o = kSampleBatch / 2; o > 0; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int g = 0; g < o; ++g) {
        const float send = up ? a[g] : a[g + o];
        const float keep = up ? a[g + o] : a[g];
        a[g] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    float ts = a[0] + __shfl_xor_sync(0xffffffffu, a[0], 16);
    const int ti = t0 + (lane & (kSampleBatch - 1));
    for (unsigned m = kmask; m; m &= m - 1) {  // the keys' weights
      const int k = __ffs(m) - 1;
      const int tk = __shfl_sync(0xffffffffu, ktile, k);
      const float cv = __shfl_sync(0xffffffffu, kcorr, k);
      if (tk == ti) ts -= cv;
    }
    ts = fmaxf(ts, 0.f);
    if (lane >= kSampleBatch || ti >= ntile) ts = 0.f;
    const FF inc = warp_ffscan(ff(ts), lane);
    const FF before = ff_add(run, ff_add(inc, -ts));  // mass before tile ti
    const unsigned h = last ? 0u : __ballot_sync(0xffffffffu, ts > 0.f && ff_gt(ff_add(before, ts), tin));
    const unsigned pz = __ballot_sync(0xffffffffu, ts > 0.f);
    const float tv = ff_add(tin, ff_neg(before)).hi;  // relative to the tile's start
    if (h) {
      const int s = __ffs(h) - 1;
      tsel = t0 + s;
      tw = __shfl_sync(0xffffffffu, tv, s);
    } else if (pz) {
      const int s = 31 - __clz(pz);
      tlast = t0 + s;
      twlast = __shfl_sync(0xffffffffu, tv, s);
    }
    run = ff_add(run, shfl(inc, 31));
  }
  if (tsel < 0) {  // rounding: U * R at or past the end of the piece
    last = true;
    tsel = tlast;
    tw = twlast;
  }
  if (tsel < 0) return -1;
  // ---- the chosen tile: an fp32 scan of its lanes relative to its start,
  // then the crossing lane walks its vector --------------------------------
  const int j = tsel * 32 + lane;
  float r[VW];
#pragma unroll
  for (int k = 0; k < VW; ++k) r[k] = 0.f;
  if (j < nvc) rvals(load_vec<DT, true>(row, e0, e1, j), j, r);
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
  const unsigned hl = last ? 0u : __ballot_sync(0xffffffffu, vs > 0.f && inc > tw);
  const unsigned pl = __ballot_sync(0xffffffffu, vs > 0.f);
  const bool lastel = hl == 0;  // past the end, or rounding inside the tile
  const int sel = hl ? __ffs(hl) - 1 : (pl ? 31 - __clz(pl) : -1);
  int tok = -1;
  float rt = 0.f;
  bool kfb = false;
  if (lane == sel) {
    float runv = lane > 0 ? exc : 0.f;
    int kk = -1, kl = -1;
#pragma unroll
    for (int k = 0; k < VW; ++k)
      if (r[k] > 0.f) {
        runv += r[k];
        kl = k;
        if (!lastel && kk < 0 && runv > tw) kk = k;
      }
    const int ksel = kk >= 0 ? kk : kl;  // rounding within the vector: its last r > 0
#pragma unroll
    for (int k = 0; k < VW; ++k)
      if (k == ksel) rt = r[k];
    tok = ksel >= 0 ? static_cast<int>(e0 + static_cast<int64_t>(j) * VW + ksel) : -1;
    kfb = kk < 0;
  }
  if (sel < 0) return -1;
  tok = __shfl_sync(0xffffffffu, tok, sel);
  rt = __shfl_sync(0xffffffffu, rt, sel);
  fb = last || __shfl_sync(0xffffffffu, kfb, sel);
  q = __fdiv_rn(rt, R.hi);
  return tok;
}

// The sampler's outputs for row b: its token, sigma(token), and its status.
__device__ __forceinline__ void sample_write(const DecideParams& P, int b, int64_t u0, int status,
                                             int32_t token, float q) {
  const bool ok = !(status & kErrors);
  P.out_tokens[u0] = ok ? token : -1;
  if (P.q_draft) P.q_draft[b] = ok ? q : 0.f;
  if (P.row_status) P.row_status[b] = ok ? (status & kFallback) : (status & kErrors);
}

// One warp per sampled row (rows 8 x blockIdx.x + warp); aligned rows whose
// records carry their chunks' pieces (P.pieces > 0).  Dynamic shared memory: the
// segment sums of one whole row for the CTA-wide pass.
template <int DT>
__global__ void __launch_bounds__(kThreads, 2) sample_rows_kernel(const DecideParams P) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  extern __shared__ float segs[];  // [tiles * kWarps] of one row, for the CTA-wide pass
  __shared__ WarpKeys wkeys[kWarps];
  __shared__ PendRow pend[kWarps];
  __shared__ int32_t npend[kWarps];
  __shared__ FF total;
  __shared__ FF tau_s;
  __shared__ int32_t pass_again, mode_s;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int b = static_cast<int>(blockIdx.x) * kWarps + warp;
  const bool active = b < P.B;
  if (lane == 0) npend[warp] = 0;

  if (active) {
    const RowCtx X = row_ctx<kModeSample>(P, b);
    const float U = P.unif[X.L.u_off + X.u_draw];
    const char* row = static_cast<const char*>(P.zd) + X.L.d_off * E::ES;
    // the records and candidates are the previous kernel's output
    pdl_wait_primary();
    // ---- 1. the row's statistics ---------------------------------------------
    const PosStats ps = combine_position<32>(P.recs + X.u0 * P.nchunk, P.nchunk, X.c, lane);
    // ---- 2. its top-F_s keys, their mass and the F_s-th key -----------------
    float d = 0.f;
    SgW w{1.f, pos_inf(), -1};
    int nk = 0;
    if (X.sg_on) {
      const int ncand = static_cast<int>(P.nchunk) * P.F;
      const WarpTopF Lk = warp_keys(P.cand_v + X.u0 * ncand, P.cand_i + X.u0 * ncand, ncand, P.F, lane,
                                    wkeys[warp]);
      const int fs = P.sg_F;
      d = (lane < fs && Lk.i != INT_MAX) ? ex2((Lk.v - ps.Md) * X.c) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      // the F_s-th key (with F_s = 0 none: every logit sits above -inf, and C = 1)
      const float zl = __shfl_sync(0xffffffffu, Lk.v, fs > 0 ? fs - 1 : 0);
      const int32_t il = __shfl_sync(0xffffffffu, Lk.i, fs > 0 ? fs - 1 : 0);
      w = fs > 0 ? SgW{P.sg_C, zl, il} : SgW{P.sg_C, neg_inf(), -1};
      const bool valid = lane < fs && Lk.i != INT_MAX;
      if (valid) {  // the keys, for the pieces' masses (after the merge's last use of the scratch)
        wkeys[warp].ov[lane] = Lk.v;
        wkeys[warp].oi[lane] = Lk.i;
      }
      nk = __popc(__ballot_sync(0xffffffffu, valid));
      __syncwarp();
    }
    // ---- 3. the checks and the weighted normaliser ---------------------------
    const FF one_m_c = two_sum(1.f, -w.C);
    const FF sdp = X.sg_on ? ff_add(ps.Sd, ff_neg(ff_mul(one_m_c, d))) : ps.Sd;
    int status = X.temp_ok ? 0 : kBadTemp;
    if (X.kb_in < 0) status |= kBadCount;
    if (X.temp_ok && (X.greedy ? ((ps.bad & 1) || ps.id == INT_MAX)
                               : (!(ps.Sd.hi >= 1.f) || ps.Md == kNegMax || !(sdp.hi > 0.f))))
      status |= kNonFinite;
    if (ps.bad & 2) status |= kTimeout;
    const bool ok = !(status & kErrors);
    if (!ok || X.greedy) {
      if (lane == 0) sample_write(P, b, X.u0, status, ok ? ps.id : -1, ok ? 1.f : 0.f);
    } else if (X.sg_on && __fmul_rn(one_m_c.hi, d) > 0.5f * ps.Sd.hi) {
      // the keys hold most of the mass: the CTA-wide pass over the whole row
      if (lane == 0) {
        npend[warp] = 1;
        pend[warp] = PendRow{row, ps.Md, X.c, __fdiv_rn(1.f, sdp.hi), U, w, status, b, X.u0};
      }
    } else {
      // ---- 4-5. the piece holding U * R -----------------------------------------
      float q;
      bool fb;
      const int tok = warp_piece_draw<DT>(P.piece_stats + X.u0 * P.nchunk * kMaxPieces, P.nchunk, P.chunk,
                                          P.pieces, P.V, ps.Md, X.c,
                                         row, U, wkeys[warp].ov, wkeys[warp].oi, nk, w, q, fb);
      if (lane == 0) sample_write(P, b, X.u0, status | (fb ? kFallback : 0), tok, q);
    }
  }
  __syncthreads();

  // ---- the CTA-wide pass, one pending row after another ---------------------
  const int nv = (P.V + VW - 1) / VW;
  const int ntl = (nv + kThreads - 1) / kThreads;
  for (int pw = 0; pw < kWarps; ++pw) {
    if (!npend[pw]) continue;  // (the same in every thread)
    const PendRow& R = pend[pw];
    if (threadIdx.x == 0) mode_s = 3;
    __syncthreads();
    for (int pass = 0; pass < 2; ++pass) {
      const int mode = mode_s;
      for (int t0 = 0; t0 < ntl; t0 += kTileUnroll) {
        float s[kTileUnroll];
#pragma unroll
        for (int g = 0; g < kTileUnroll; ++g) {
          const int j = (t0 + g) * kThreads + threadIdx.x;
          s[g] = 0.f;
          if (j < nv) {
            float r[VW];
            residual_vec<DT, true>(R.row, nullptr, 0, P.V, j, mode, R.mt, R.mt, R.c, R.ist, R.ist, -1,
                                   R.w, r);
#pragma unroll
            for (int k = 0; k < VW; ++k) s[g] += r[k];
          }
        }
#pragma unroll
        for (int g = 0; g < kTileUnroll; ++g) {
          const float ws = warp_sum(s[g]);
          if (lane == 0 && t0 + g < ntl) segs[(t0 + g) * kWarps + warp] = ws;
        }
      }
      __syncthreads();
      if (warp == 0) {
        FF acc = ff(0.f);
        for (int sg = lane; sg < ntl * kWarps; sg += 32) acc = ff_add(acc, segs[sg]);
        acc = warp_ffsum_all(acc);
        if (lane == 0) {
          total = acc;
          tau_s = ff_mul(acc, R.U);
          pass_again = 0;
          if (!(acc.hi > 0.f) && mode == 3) {  // zero weighted mass: draw from p instead
            mode_s = 1;
            pass_again = 1;
          }
        }
      }
      __syncthreads();
      if (!pass_again) break;
    }
    if (warp == 0) {
      const FF Rt = total;
      int status = R.status;
      if (mode_s == 1) status |= kFallback;
      int tok = -1;
      float rq = 0.f;
      if (Rt.hi > 0.f) {
        // U * R at or past the end after rounding: the last index with r > 0
        const bool lp = !ff_gt(Rt, tau_s);
        if (lp) status |= kFallback;
        tok = owner_scan<DT, true>(segs, ntl, tau_s, ff(0.f), lp, R.row, nullptr, 0, P.V, nv, mode_s, R.mt,
                                   R.mt, R.c, R.ist, R.ist, -1, R.w, rq);
      }
      if (lane == 0)
        sample_write(P, R.b, R.u0, status, tok,
                     Rt.hi > 0.f ? __fdiv_rn(rq, Rt.hi) : 0.f);
    }
    __syncthreads();
  }
}

}  // namespace specv
