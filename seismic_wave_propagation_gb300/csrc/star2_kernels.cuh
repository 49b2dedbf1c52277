// Two sweeps of the 7-point (radius 1) star stencil in one pass over the grid (temporal
// blocking of the ping-pong loop): u2 = S(S(u0)), with the shell of every level fixed to
// u0's.  The intermediate level u1 never leaves the SM.  Every thread owns a float4
// column of NR consecutive rows in both stages (NR = 2: 256 threads; NR = 4: 128).
//
// The plane loop is the 2.5D stream of the one-sweep kernel ("Accelerating High-Order
// Stencils on GPUs", 2.5D blocking with a register window along z), run twice per landed
// plane:
//   * stage 1: plane p of u0 lands in the shared ring (TMA).  Each thread runs the
//     first sweep's z filter on its own columns (transposed form, two partial sums) and
//     adds the in-plane terms of plane p; the first-sweep value u1 at plane p-1 is then
//     complete.  Stage 1 covers the output tile plus one point on every side (rows
//     y0-1 .. y0+TY, columns x0-1 .. x0+64: the extra columns by the two threads at the
//     ends of each row group).  Points on a face of the grid take u0's value (fixed
//     shell).  The result goes into one of two shared u1 planes.
//   * after one CTA barrier per plane, stage 2 runs the second sweep on u1 in the same
//     way and emits u2 at plane p-2.
// So each plane of u0 is read from DRAM once and each plane of u2 written once per two
// sweeps; the cost is the first sweep's ring of extra points (about 10 %) and the barrier.
#pragma once

#include "star_kernels.cuh"

namespace libstencil {

template <int STAGES, int NR = 2>
struct Star2Cfg {
  static constexpr int TY = 30;            // output rows of the second sweep per tile
  static constexpr int BW = kTX + 2 * kHX; // 72: staged x range x0-4 .. x0+67
  static constexpr int BH = TY + 4;        // 34: staged rows y0-2 .. y0+31
  static constexpr int UH = TY + 2;        // 32: first-sweep rows y0-1 .. y0+30
  static_assert(UH % NR == 0, "row groups tile the first-sweep rows");
  static constexpr int kGroups = UH / NR;  // row groups of NR rows
  static constexpr int kThreads = 16 * kGroups;  // 16 column groups x the row groups
  // Second sweep: the groups whose first row is inside the tile; the last may run past
  // its end (NR = 4: rows 28-31 of 30) and read u1 rows up to UH + 1, which are kept zero
  // (their outputs are never stored).
  static constexpr int kActive2 = (TY + NR - 1) / NR;
  static constexpr int kU1Rows = NR * (kActive2 - 1) + NR + 2 > UH ? NR * (kActive2 - 1) + NR + 2 : UH;
  static constexpr int kPlaneBytes = BW * BH * 4;
  static constexpr int kPlaneStride = (kPlaneBytes + 127) / 128 * 128;
  static constexpr int kU1Floats = BW * kU1Rows;
  static constexpr int kCurOff = (8 * STAGES + 15) / 16 * 16;
  static constexpr int kIssOff = kCurOff + (int)sizeof(Cursor);
  static constexpr int kRingOffset = (kIssOff + 4 * STAGES + 127) / 128 * 128;
  static constexpr int kU1Offset = kRingOffset + STAGES * kPlaneStride;
  static constexpr int kSmemBytes = kU1Offset + 2 * kU1Floats * 4;
  static constexpr int kLookahead = STAGES - 1;
  static_assert(kLookahead >= 1, "ring needs a plane in flight");
  static_assert((BW * 4) % 16 == 0 && BW <= 256 && BH <= 256, "TMA box");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// Item -> tile (x0, y0) and its L = zb - za + 4 landed planes za-2 .. zb+1: two fill
// planes per sweep on each side of the chunk's output planes [za, zb).
template <int TY>
__device__ __forceinline__ void item2_geometry(const StarParams& p, int item, int& x0, int& y0, int& L,
                                               int& zs) {
  int b = 0;
  while (b + 1 < p.nboxes && item >= p.box[b + 1].item0) ++b;
  const Box& q = p.box[b];
  const int local = item - q.item0;
  const int chunk = local / q.ntiles;
  const int tile = local - chunk * q.ntiles;
  const int by = tile / q.ntx;
  const int bx = tile - by * q.ntx;
  x0 = (q.tx0 + bx) * kTX;
  y0 = 1 + (q.ty0 + by) * TY;
  const int za = q.z0 + (int)(((long long)chunk * q.nzi) / q.nchunks);
  const int zb = q.z0 + (int)(((long long)(chunk + 1) * q.nzi) / q.nchunks);
  L = zb - za + 4;
  zs = za - 2;
}

template <int TY>
__device__ __forceinline__ void cursor2_set_item(const StarParams& p, Cursor& k, int item) {
  k.item = item;
  k.j = 0;
  k.dz = 1;
  if (item < p.nitems) item2_geometry<TY>(p, item, k.x0, k.y0, k.L, k.zs);
}

template <int TY>
__device__ __forceinline__ void cursor2_advance(const StarParams& p, Cursor& k) {
  if (++k.j == k.L) cursor2_set_item<TY>(p, k, k.item + (int)gridDim.x);
}

__device__ __forceinline__ bool on_face(const StarParams& p, int x, int y) {
  return x == 0 || x == p.nx - 1 || y == 0 || y == p.ny - 1;
}

template <int STAGES, int MINB, int NR>
__global__ void __launch_bounds__(Star2Cfg<STAGES, NR>::kThreads, MINB)
    star2_sweep_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap,
                       const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                       const __grid_constant__ CUtensorMap, const __grid_constant__ StarParams p) {
  using C = Star2Cfg<STAGES, NR>;
  constexpr int TY = C::TY;
  constexpr int BW = C::BW;
  constexpr int PSTRIDE = C::kPlaneStride / 4;
  constexpr int NWARPS = C::kThreads / 32;

  extern __shared__ __align__(128) unsigned char smem[];
  Cursor* cur = reinterpret_cast<Cursor*>(smem + C::kCurOff);
  int* lastld = reinterpret_cast<int*>(smem + C::kIssOff);
  const uint32_t base = smem_addr(smem);
  const uint32_t ring_base = base + C::kRingOffset;
  const float* ring = reinterpret_cast<const float*>(smem + C::kRingOffset);
  float* u1buf = reinterpret_cast<float*>(smem + C::kU1Offset);

  if ((int)blockIdx.x >= p.nitems) return;

  const int tid = threadIdx.x;
  const int tc = tid & 15;         // column group: x0 + 4*tc .. +3
  const int tr = tid >> 4;         // row group
  const int col = 4 * tc;
  const bool leader = tid == 0;
  const int warp = tid >> 5;
  const bool lane0 = (tid & 31) == 0;
  // Stage 1 rows y0-1+NR*tr+k (k < NR): staged rows NR*tr+1+k; u1 rows NR*tr+k.
  const int own1 = (NR * tr + 1) * BW + kHX + col;
  const int w1 = NR * tr * BW + kHX + col;
  // Stage 2 rows y0+NR*tr+k (groups starting inside the tile): u1 rows NR*tr+1+k.
  const int own2 = (NR * tr + 1) * BW + kHX + col;
  const bool st2 = NR * tr < TY;
  constexpr unsigned kKeepAll = (1u << (5 * NR)) - 1u;  // every point of a thread on a face
  // The threads at both ends of a row group also compute the first sweep one column
  // beyond the tile: x0-1 (staged column kHX-1) and x0+64 (kHX+kTX).
  const bool ext = tc == 0 || tc == 15;
  const int ecol = tc == 0 ? kHX - 1 : kHX + kTX;

  auto produce_u = [&](int counter) {
    Cursor& k = cur[0];
    if (k.item >= p.nitems) return;
    const int slot = counter % STAGES;
    const uint32_t bar = base + 8u * slot;
    lastld[slot] = counter;
    if (counter != p.debug_skip) {
      mbar_arrive_expect_tx(bar, C::kPlaneBytes);
      tma_load_3d(ring_base + slot * C::kPlaneStride, &tm_u, bar, k.x0 - kHX, k.y0 - 2, k.zs + k.j);
    }
    ++k.issued;
    cursor2_advance<TY>(p, k);
  };

  const bool bad_smem = (base & 127u) != 0u;
  if constexpr (C::kU1Rows > C::UH) {  // the u1 rows past the first sweep's stay zero
    constexpr int kTail = (C::kU1Rows - C::UH) * BW;
    for (int i = tid; i < 2 * kTail; i += C::kThreads)
      u1buf[(i / kTail) * C::kU1Floats + C::UH * BW + i % kTail] = 0.f;
  }
  if (leader) {
    if (bad_smem) atomicOr(p.status, kStatusBadSmem);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(base + 8u * s, 1);
      lastld[s] = -1;
    }
    fence_mbar_init();
    cursor2_set_item<TY>(p, cur[0], blockIdx.x);
    cur[0].issued = 0;
  }
  if (__syncthreads_or(bad_smem)) return;
  if (leader)
    for (int c = 0; c <= C::kLookahead; ++c) produce_u(c);

  bool failed = false;
  auto fail = [&](int counter) {
    if (atomicOr(p.status, kStatusTimeout) == 0u) {
      p.status[1] = blockIdx.x;
      p.status[2] = (unsigned)counter;
    }
    failed = true;
  };

  const float2 c0 = make_float2(p.c[0], p.c[0]);
  const float2 c1 = make_float2(p.c[1], p.c[1]);
  const P4 zero = P4{make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  P4 s1[2][NR], s2[2][NR], xprev[NR];  // z-filter partial sums of both sweeps; u0 of the last plane
  float es1[2][NR], eprev[NR];         // the same for the extra column
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    s1[0][k] = s1[1][k] = s2[0][k] = s2[1][k] = xprev[k] = zero;
    es1[0][k] = es1[1][k] = eprev[k] = 0.f;
  }

  int J = 0, slot = 0, pwarp = 0, ub = 0;
  uint32_t phase = 0;
  const size_t plane = (size_t)p.nx * p.ny;
  for (int item = blockIdx.x; item < p.nitems; item += gridDim.x) {
    int x0, y0, L, zs;
    item2_geometry<TY>(p, item, x0, y0, L, zs);
    const int gx = x0 + col;
    const int gxe = tc == 0 ? x0 - 1 : x0 + kTX;
    int gy1[NR], gy2[NR];
    bool row_ok[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      gy1[k] = y0 - 1 + NR * tr + k;
      gy2[k] = y0 + NR * tr + k;
      row_ok[k] = st2 && NR * tr + k < TY && gy2[k] < p.ny - 1 && gx < p.nx;
    }
    const bool vec_ok = gx >= 1 && gx + 4 <= p.nx - 1;
    // Which of this thread's first-sweep points lie on an x or y face (bit 4k + e; the
    // extra column's point of row k: bit 4 NR + k): fixed for the whole item.
    unsigned face = 0u;
#pragma unroll
    for (int k = 0; k < NR; ++k) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (on_face(p, gx + e, gy1[k])) face |= 1u << (4 * k + e);
      if (ext && on_face(p, gxe, gy1[k])) face |= 1u << (4 * NR + k);
    }
    for (int j = 0; j < L; ++j) {
      if (!mbar_wait_bounded(base + 8u * slot, phase)) fail(J);
      const float* pl = ring + slot * PSTRIDE;
      const int pz = zs + j;  // the landed plane
      P4 x[NR];
      float ex[NR];
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        x[k] = ldp4(pl + own1 + k * BW);
        ex[k] = 0.f;
      }
      if (ext) {
#pragma unroll
        for (int k = 0; k < NR; ++k) ex[k] = pl[(NR * tr + 1 + k) * BW + ecol];
      }
      float* u1w = u1buf + ub * C::kU1Floats;

      // ---- stage 1: u1 at plane pz-1 is complete, write it --------------------------------
      if (j >= 2) {
        // Points on a face keep u0: the whole plane on a z face, else the masked points.
        const unsigned keep = (pz - 1 == 0 || pz - 1 == p.nz - 1) ? kKeepAll : face;
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          P4 v = fma2x(c1, x[k], s1[0][k]);
          if (keep) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (keep & (1u << (4 * k + e))) pset(v, e, pget(xprev[k], e));
          }
          *reinterpret_cast<float4*>(u1w + w1 + k * BW) = tof4(v);
        }
        if (ext) {
#pragma unroll
          for (int k = 0; k < NR; ++k) {
            float v = fmaf(c1.x, ex[k], es1[0][k]);
            if (keep & (1u << (4 * NR + k))) v = eprev[k];
            u1w[(NR * tr + k) * BW + ecol] = v;
          }
        }
      }
      // In-plane terms of plane pz, whose u1 is needed (planes za-1 .. zb).
      if (j >= 1 && j <= L - 2) {
        const P4 up = ldp4(pl + own1 - BW);       // row above the group
        const P4 dn = ldp4(pl + own1 + NR * BW);  // row below the group
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          const float* rowp = pl + own1 + k * BW;
          const P4& yn = k == 0 ? up : x[k > 0 ? k - 1 : 0];
          const P4& ys = k == NR - 1 ? dn : x[k < NR - 1 ? k + 1 : 0];
          P4& a = s1[1][k];
          a.a = __ffma2_rn(c1, __fadd2_rn(yn.a, ys.a), a.a);
          a.b = __ffma2_rn(c1, __fadd2_rn(yn.b, ys.b), a.b);
          const float l = rowp[-1], r = rowp[4];
          pset(a, 0, fmaf(c1.x, l + pget(x[k], 1), pget(a, 0)));
          pset(a, 1, fmaf(c1.x, pget(x[k], 0) + pget(x[k], 2), pget(a, 1)));
          pset(a, 2, fmaf(c1.x, pget(x[k], 1) + pget(x[k], 3), pget(a, 2)));
          pset(a, 3, fmaf(c1.x, pget(x[k], 2) + r, pget(a, 3)));
        }
        if (ext) {
#pragma unroll
          for (int k = 0; k < NR; ++k) {
            const float* q = pl + (NR * tr + 1 + k) * BW + ecol;
            es1[1][k] = fmaf(c1.x, (q[-1] + q[1]) + (q[-BW] + q[BW]), es1[1][k]);
          }
        }
      }
      // z filter of the first sweep: every partial sum moves one slot down.
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        s1[0][k] = fma2x(c0, x[k], s1[1][k]);
        s1[1][k] = P4{__fmul2_rn(c1, x[k].a), __fmul2_rn(c1, x[k].b)};
        es1[0][k] = fmaf(c0.x, ex[k], es1[1][k]);
        es1[1][k] = c1.x * ex[k];
        xprev[k] = x[k];
        eprev[k] = ex[k];
      }

      // ---- the CTA meets: u1 of plane pz-1 is in shared memory, the slot is free ---------
      ++J;
      if (++slot == STAGES) {
        slot = 0;
        phase ^= 1u;
      }
      const bool stop = __syncthreads_or(failed) != 0;
      if (lane0 && !stop && warp == pwarp) {
        fence_proxy_async_smem();
        produce_u(J - 1 + STAGES);
      }
      if (++pwarp == NWARPS) pwarp = 0;
      if (stop) goto drain;

      // ---- stage 2: the second sweep on u1 --------------------------------------------------
      if (j >= 2 && st2) {
        const float* u1r = u1buf + ub * C::kU1Floats;
        P4 w[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) w[k] = ldp4(u1r + own2 + k * BW);
        if (j >= 4) {  // u2 at plane pz-2
          float* const oz = p.out + (size_t)(pz - 2) * plane + gx;
#pragma unroll
          for (int k = 0; k < NR; ++k) {
            const P4 o = fma2x(c1, w[k], s2[0][k]);
            if (row_ok[k]) {
              float* dst = oz + (size_t)gy2[k] * p.nx;
              if (vec_ok) {
                __stcs(reinterpret_cast<float4*>(dst), tof4(o));
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (gx + e >= 1 && gx + e < p.nx - 1) dst[e] = pget(o, e);
              }
            }
          }
        }
        if (j >= 3 && j <= L - 2) {  // in-plane terms of u1 plane pz-1, an output plane
          const P4 up = ldp4(u1r + own2 - BW);
          const P4 dn = ldp4(u1r + own2 + NR * BW);
#pragma unroll
          for (int k = 0; k < NR; ++k) {
            const float* rowp = u1r + own2 + k * BW;
            const P4& yn = k == 0 ? up : w[k > 0 ? k - 1 : 0];
            const P4& ys = k == NR - 1 ? dn : w[k < NR - 1 ? k + 1 : 0];
            P4& a = s2[1][k];
            a.a = __ffma2_rn(c1, __fadd2_rn(yn.a, ys.a), a.a);
            a.b = __ffma2_rn(c1, __fadd2_rn(yn.b, ys.b), a.b);
            const float l = rowp[-1], r = rowp[4];
            pset(a, 0, fmaf(c1.x, l + pget(w[k], 1), pget(a, 0)));
            pset(a, 1, fmaf(c1.x, pget(w[k], 0) + pget(w[k], 2), pget(a, 1)));
            pset(a, 2, fmaf(c1.x, pget(w[k], 1) + pget(w[k], 3), pget(a, 2)));
            pset(a, 3, fmaf(c1.x, pget(w[k], 2) + r, pget(a, 3)));
          }
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
          s2[0][k] = fma2x(c0, w[k], s2[1][k]);
          s2[1][k] = P4{__fmul2_rn(c1, w[k].a), __fmul2_rn(c1, w[k].b)};
        }
      }
      ub ^= 1;
    }
  }
  return;

drain:
  // A wait ran out: wait (bounded) for the last copy issued into each slot, then leave.
  if (leader) {
    for (int sl = 0; sl < STAGES; ++sl) {
      const int c = lastld[sl];
      if (c >= 0 && c != p.debug_skip && !mbar_wait_bounded(base + 8u * sl, (c / STAGES) & 1))
        atomicOr(p.status, kStatusDrainTimeout);
    }
  }
  __syncthreads();
}

}  // namespace libstencil
