// Star-stencil sweep kernels for sm_103a (GB300): 2.5D blocking with TMA staging.
//
// What is computed (radius R, fp32, flat grid with x innermost):
//   out(x,y,z) = c0*u + sum_{r=1..R} c_r*(u(x±r,y,z) + u(x,y±r,z) + u(x,y,z±r))
// at every point at least R away from every face; optionally fused with the acoustic
// update u_next = (2u - (1-eta) u_prev + v2dt2*lap) / (1+eta).
//
// How ("Accelerating High-Order Stencils on GPUs", 2.5D blocking: a 2D x-y tile streams
// through z, the z neighbours of a thread's points never leave its registers):
//   * One CTA owns a 64 x TY output tile of the x-y plane and a contiguous range of z
//     (a "chunk").  Work items (tile, chunk) are dealt round-robin to a persistent grid in
//     z-major order, so CTAs working on neighbouring tiles march through the same planes
//     at the same time and their halos are served from L2.
//   * Each plane's (64+8) x (TY+2R) box is staged into a shared-memory ring by TMA
//     (cp.async.bulk.tensor.3d), completion tracked by an mbarrier per slot (expect-tx
//     bytes).  The CTA meets at one barrier every KB planes; right after it, lane 0 of one
//     warp (the duty rotates over the warps) refills the slots released since the last
//     one.  With DRIFT (sweeps of radius 1-3) there is no barrier: each warp counts itself
//     off a slot in shared memory when done with it, and the last one refills it, so the
//     warps drift apart by up to the ring's lookahead.
//     Out-of-range box parts are zero-filled by the TMA unit and only ever feed outputs
//     that are masked off.
//   * Every thread owns a 4 x TYT block of output columns (one float4 per row).  Along z
//     it runs the symmetric 2R+1-tap filter h_i = c_|i-R| in transposed form: when plane
//     p lands, its own values x update 2R running partial sums,
//         y = h_0 x + s_1,   s_i <- h_i x + s_{i+1} (i < 2R),   s_2R <- h_2R x,
//     and y is the z part of the output at plane p-R.  Each FMA also moves a partial sum
//     one slot down, so the z window needs no register moves and no unrolling.  The
//     in-plane part of plane p's outputs (x and y neighbours, read from the landed box)
//     is added to s_R, which emerges R planes later.  The stencil sweep therefore needs
//     only the lead plane in shared memory; the wave step keeps R more planes for u(z),
//     and so does the semi-stencil form (SEMI), which reads the centre and one half of
//     the z stencil from those planes and carries the other half in R partial sums.
//   * Every wait on an mbarrier is bounded (about 2 s).  When it runs out the kernel
//     records an error in the status block, waits (bounded) for its own copies still in
//     flight and returns; the host reads the status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace libstencil {

constexpr int kTX = 64;             // output tile width in x (floats)
constexpr int kThreadsX = kTX / 4;  // one float4 column group per thread
constexpr int kHX = 4;              // staged x halo per side; keeps the TMA x start 16-B aligned

constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusDrainTimeout = 2u;
constexpr unsigned kStatusBadSmem = 4u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// A box of work: a rectangle of output tiles times a range of output planes, cut into
// z-chunks; every (tile, chunk) pair is one work item.
struct Box {
  int tx0, ty0;     // first tile along x and y
  int ntx;          // tiles along x
  int ntiles;       // tiles in the rectangle
  int z0;           // first output plane
  int nzi;          // output planes
  int nchunks;      // z-chunks per tile column
  int item0;        // index of the box's first work item
};

constexpr int kMaxBoxes = 6;

struct StarParams {
  int nx, ny, nz;
  int nboxes;       // boxes of this launch (one for a whole-grid sweep or step)
  int nitems;       // work items of all boxes
  Box box[kMaxBoxes];
  float c[5];       // c[0] total centre weight, c[r] per-neighbour weight
  float* out;       // stencil output, or u_next for the wave step
  unsigned* status; // [0] flags, [1] block, [2] load counter of the first failure
  int debug_skip;   // load counter every CTA skips (watchdog test); -1 = none
};

// Producer cursor: the next load of the CTA's sequence (kept in shared memory; the warps
// that refill the ring take turns, and the CTA barrier between turns orders them).
struct Cursor {
  int item, j, L, x0, y0, zs, issued, dz;  // plane landed at step j: zs + dz * j
};

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, bool SEMI = false,
          int TSTORE = 0, int KB = 1>
struct StarCfg {
  static constexpr int kThreads = kThreadsX * NWY;
  static constexpr int TY = TYT * NWY;  // output tile height
  static constexpr int BW = kTX + 2 * kHX;
  static constexpr int BH = TY + 2 * R;
  static constexpr int kPlaneBytes = BW * BH * 4;  // bytes one u box transfers
  static constexpr int kPlaneStride = (kPlaneBytes + 127) / 128 * 128;
  static constexpr int kAuxFieldBytes = kTX * TY * 4;
  static constexpr int kAuxStageBytes = 3 * kAuxFieldBytes;
  static constexpr int kNumBars = STAGES + (WAVE ? ASTAGES : 0);
  static constexpr int kCurOff = (8 * kNumBars + 15) / 16 * 16;
  static constexpr int kCntOff = kCurOff + 2 * (int)sizeof(Cursor);  // release counters
  static constexpr int kIssOff = kCntOff + 4 * kNumBars;                // last load per slot
  static constexpr int kRingOffset = (kIssOff + 4 * kNumBars + 127) / 128 * 128;
  static constexpr int kAuxOffset = kRingOffset + STAGES * kPlaneStride;
  static constexpr int kStgOffset = kAuxOffset + (WAVE ? ASTAGES * kAuxStageBytes : 0);
  static constexpr int kStgPlaneBytes = kTX * TY * 4;  // one output tile, staged for a TMA store
  // TSTORE > 0: output tiles go out by TMA store from TSTORE * KB staging tiles, so that
  // the stores of the last TSTORE - 1 barrier intervals may still be reading theirs.
  static constexpr int kStgPlanes = TSTORE * KB;
  static constexpr int kSmemBytes = kStgOffset + kStgPlanes * kStgPlaneBytes;
  static constexpr int XO = TSTORE ? R : 0;  // x of the first tile's first output
  static constexpr int KEEP = (WAVE || SEMI) ? R : 0;   // planes kept behind the lead
  static constexpr int kLookahead = STAGES - KEEP - 1;  // planes in flight beyond the lead
  static_assert(kLookahead >= 1, "ring must hold the kept planes plus one in flight");
  static_assert(BW <= 256 && BH <= 256, "TMA box dimensions are limited to 256");
  static_assert((BW * 4) % 16 == 0, "TMA inner box bytes must be a multiple of 16");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  // TMA-stored tiles start at the interior origin x = R; the staged input box then starts
  // at x = R - kHX, which must be 0 for its x coordinate to stay 16-byte aligned.
  static_assert(!TSTORE || R == kHX, "TMA stores of the output need R == 4");
  static_assert(TSTORE == 0 || TSTORE >= 2, "TMA stores stage at least two barrier intervals");
};

// ---- PTX wrappers ------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete; false after ~kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  return false;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Bulk tensor store of a staged tile (shared -> global through the TMA unit), tracked in
// the issuing thread's bulk groups.  Parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All but the issuing thread's N most recent bulk-store groups have finished reading
// shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// The issuing thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float4 lds4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Four consecutive x values as two register pairs, for the packed fp32x2 arithmetic of
// sm_100-family SMs (one FFMA2 performs two FMAs in one issue slot).
struct P4 {
  float2 a, b;  // (x0, x0+1), (x0+2, x0+3)
};

__device__ __forceinline__ P4 ldp4(const float* p) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  return P4{make_float2(v.x, v.y), make_float2(v.z, v.w)};
}

__device__ __forceinline__ float4 tof4(const P4& v) { return make_float4(v.a.x, v.a.y, v.b.x, v.b.y); }

__device__ __forceinline__ P4 fma2x(const float2& c, const P4& x, const P4& y) {
  return P4{__ffma2_rn(c, x.a, y.a), __ffma2_rn(c, x.b, y.b)};
}

__device__ __forceinline__ float pget(const P4& v, int e) {
  return e == 0 ? v.a.x : e == 1 ? v.a.y : e == 2 ? v.b.x : v.b.y;
}

__device__ __forceinline__ void pset(P4& v, int e, float x) {
  if (e == 0) v.a.x = x;
  else if (e == 1) v.a.y = x;
  else if (e == 2) v.b.x = x;
  else v.b.y = x;
}

__device__ __forceinline__ float get(const float4& v, int e) {
  return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// ---- work decomposition -------------------------------------------------------------

// Item -> output tile (x0, y0), its L = zb - za + 2R landed planes and their order: the
// plane landed at step j is zs + dz * j, the output plane completed at step j >= 2R is
// zs + dz * (j - R).  Every chunk marches up (dz = 1) from za - R; the z filter is
// symmetric, so a chunk marching down from zb + R - 1 (dz = -1) would compute the same.
template <int R, int TY, int XO>
__device__ __forceinline__ void item_geometry(const StarParams& p, int item, int& x0, int& y0,
                                              int& L, int& zs, int& dz) {
  int b = 0;
  while (b + 1 < p.nboxes && item >= p.box[b + 1].item0) ++b;
  const Box& q = p.box[b];
  const int local = item - q.item0;
  const int chunk = local / q.ntiles;
  const int tile = local - chunk * q.ntiles;
  const int by = tile / q.ntx;
  const int bx = tile - by * q.ntx;
  x0 = XO + (q.tx0 + bx) * kTX;
  y0 = R + (q.ty0 + by) * TY;
  const int za = q.z0 + (int)(((long long)chunk * q.nzi) / q.nchunks);
  const int zb = q.z0 + (int)(((long long)(chunk + 1) * q.nzi) / q.nchunks);
  L = zb - za + 2 * R;
  dz = 1;
  zs = za - R;
}

template <int R, int TY, int XO>
__device__ __forceinline__ void cursor_set_item(const StarParams& p, Cursor& k, int item) {
  k.item = item;
  k.j = 0;
  if (item < p.nitems) item_geometry<R, TY, XO>(p, item, k.x0, k.y0, k.L, k.zs, k.dz);
}

template <int R, int TY, int XO>
__device__ __forceinline__ void cursor_advance(const StarParams& p, Cursor& k) {
  if (++k.j == k.L) cursor_set_item<R, TY, XO>(p, k, k.item + (int)gridDim.x);
}

// ---- the kernel ----------------------------------------------------------------------

template <int R, int TYT, int NWY, int STAGES, int ASTAGES, bool WAVE, int MINB, int KB, bool NOETA,
          bool SEMI, bool DRIFT, int TSTORE>
__global__ void __launch_bounds__(kThreadsX * NWY, MINB)
    star_sweep_kernel(const __grid_constant__ CUtensorMap tm_u,
                      const __grid_constant__ CUtensorMap tm_uprev,
                      const __grid_constant__ CUtensorMap tm_v2dt2,
                      const __grid_constant__ CUtensorMap tm_eta,
                      const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ StarParams p) {
  using C = StarCfg<R, TYT, NWY, STAGES, ASTAGES, WAVE, SEMI, TSTORE, KB>;
  static_assert(!(TSTORE && (SEMI || DRIFT)), "TMA stores: plain sweep or wave step, barrier protocol");
  static_assert(!(WAVE && SEMI), "the semi-stencil form is a plain sweep");
  static_assert(!(WAVE && DRIFT), "the wave step's aux ring needs the per-plane barrier");
  constexpr int TY = C::TY;
  constexpr int BW = C::BW;
  constexpr int KEEP = C::KEEP;
  constexpr int PSTRIDE = C::kPlaneStride / 4;  // floats between ring slots
  constexpr int XO = C::XO;

  extern __shared__ __align__(128) unsigned char smem[];
  Cursor* cur = reinterpret_cast<Cursor*>(smem + C::kCurOff);  // [0] u loads, [1] aux loads
  int* relcnt = reinterpret_cast<int*>(smem + C::kCntOff);     // warps done with a slot
  int* lastld = reinterpret_cast<int*>(smem + C::kIssOff);     // last load counter per slot
  const uint32_t base = smem_addr(smem);
  const uint32_t ring_base = base + C::kRingOffset;
  const uint32_t aux_base = base + C::kAuxOffset;
  const float* ring = reinterpret_cast<const float*>(smem + C::kRingOffset);
  const float* auxr = reinterpret_cast<const float*>(smem + C::kAuxOffset);
  float* stg = reinterpret_cast<float*>(smem + C::kStgOffset);  // staged output tiles (TSTORE)
  const uint32_t stg_base = base + C::kStgOffset;

  if ((int)blockIdx.x >= p.nitems) return;

  constexpr int NWARPS = C::kThreads / 32;
  const int tid = threadIdx.x;
  const int col = 4 * (tid % kThreadsX);     // x offset of this thread's float4 in the tile
  const int row0 = (tid / kThreadsX) * TYT;  // first tile row of this thread
  const int own = (row0 + R) * BW + kHX + col;  // its first point in a landed box
  const bool leader = tid == 0;
  const int warp = tid >> 5;
  const bool lane0 = (tid & 31) == 0;

  // Producer: stage the u box of the next plane in the cursor's sequence.
  auto produce_u = [&](int counter) {
    Cursor& k = cur[0];
    if (k.item >= p.nitems) return;
    const int slot = counter % STAGES;
    const uint32_t bar = base + 8u * slot;
    lastld[slot] = counter;
    if (counter != p.debug_skip) {
      mbar_arrive_expect_tx(bar, C::kPlaneBytes);
      tma_load_3d(ring_base + slot * C::kPlaneStride, &tm_u, bar, k.x0 - kHX, k.y0 - R,
                  k.zs + k.dz * k.j);
    }
    ++k.issued;
    cursor_advance<R, TY, XO>(p, k);
  };
  // Producer: stage u_prev, v2dt2, eta of the output plane of an emitting step.
  auto produce_aux = [&](int counter) {
    Cursor& k = cur[1];
    if (k.item >= p.nitems) return;
    const int slot = counter % ASTAGES;
    const uint32_t bar = base + 8u * (STAGES + slot);
    if (k.j >= 2 * R) {
      const uint32_t dst = aux_base + slot * C::kAuxStageBytes;
      const int z = k.zs + k.dz * (k.j - R);
      mbar_arrive_expect_tx(bar, (NOETA ? 2 : 3) * C::kAuxFieldBytes);
      tma_load_3d(dst, &tm_uprev, bar, k.x0, k.y0, z);
      tma_load_3d(dst + C::kAuxFieldBytes, &tm_v2dt2, bar, k.x0, k.y0, z);
      if (!NOETA) tma_load_3d(dst + 2 * C::kAuxFieldBytes, &tm_eta, bar, k.x0, k.y0, z);
    } else {
      mbar_arrive(bar);  // filling step: nothing to stage, just complete the phase
    }
    ++k.issued;
    cursor_advance<R, TY, XO>(p, k);
  };

  const bool bad_smem = (base & 127u) != 0u;  // TMA destinations need 128-B alignment
  if (leader) {
    if (bad_smem) atomicOr(p.status, kStatusBadSmem);
    for (int s = 0; s < C::kNumBars; ++s) {
      mbar_init(base + 8u * s, 1);
      relcnt[s] = 0;
      lastld[s] = -1;
    }
    fence_mbar_init();
    cursor_set_item<R, TY, XO>(p, cur[0], blockIdx.x);
    cur[0].issued = 0;
    cur[1] = cur[0];
  }
  if (__syncthreads_or(bad_smem)) return;
  if (leader) {
    for (int c = 0; c <= C::kLookahead; ++c) produce_u(c);
    if (WAVE)
      for (int c = 0; c < ASTAGES; ++c) produce_aux(c);
  }

  bool failed = false;  // this thread saw a wait run out
  auto fail = [&](int counter) {
    if (atomicOr(p.status, kStatusTimeout) == 0u) {
      p.status[1] = blockIdx.x;
      p.status[2] = (unsigned)counter;
    }
    failed = true;
  };

  // s[i][k]: partial sum of the output (i + 1 - R) planes after the current one, row k
  // (semi-stencil form: of the output R - 1 - i planes before the current one).
  constexpr int NS = SEMI ? R : 2 * R;
  P4 s[NS][TYT];
#pragma unroll
  for (int i = 0; i < NS; ++i)
#pragma unroll
    for (int k = 0; k < TYT; ++k) s[i][k] = P4{make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 cc[R + 1];  // coefficients duplicated into register pairs
#pragma unroll
  for (int r = 0; r <= R; ++r) cc[r] = make_float2(p.c[r], p.c[r]);

  int J = 0;               // load counter of the current step
  int slot = 0;            // J % STAGES
  uint32_t phase = 0;      // (J / STAGES) & 1
  int aslot = 0;           // J % ASTAGES
  uint32_t aphase = 0;     // (J / ASTAGES) & 1
  int pwarp = 0;           // the warp that refills the ring at the next barrier
  int since = 0;           // steps since the last CTA barrier (one barrier per KB planes)
  int stg_slot = 0;        // staging tile of the next output plane (TSTORE)
  int emitted = 0;         // output planes staged since the last barrier (TSTORE)
  const size_t plane = (size_t)p.nx * p.ny;
  for (int item = blockIdx.x; item < p.nitems; item += gridDim.x) {
    int x0, y0, L, zs, dz;
    item_geometry<R, TY, XO>(p, item, x0, y0, L, zs, dz);  // L planes land in turn
    const int gx = x0 + col;
    const int gy0 = y0 + row0;
    // Output masks and row addresses of this thread, fixed for the whole item.
    const bool vec_ok = gx >= R && gx + 4 <= p.nx - R;
    bool row_ok[TYT];
#pragma unroll
    for (int k = 0; k < TYT; ++k) row_ok[k] = gy0 + k < p.ny - R && gx < p.nx;
    float* const orow = p.out + (size_t)gy0 * p.nx + gx;
    for (int j = 0; j < L; ++j) {
      if (!mbar_wait_bounded(base + 8u * slot, phase)) fail(J);
      const float* pl = ring + slot * PSTRIDE;
      P4 xv[TYT];
#pragma unroll
      for (int k = 0; k < TYT; ++k) xv[k] = ldp4(pl + own + k * BW);

      if (j >= 2 * R) {
        // Output plane z = (landed plane) - R is complete once its z part is added.
        const int z = zs + dz * (j - R);
        P4 o[TYT];
#pragma unroll
        for (int k = 0; k < TYT; ++k) o[k] = fma2x(cc[R], xv[k], s[0][k]);
        if constexpr (WAVE) {
          if (!mbar_wait_bounded(base + 8u * (STAGES + aslot), aphase)) fail(J);
          const float* pa = auxr + aslot * (C::kAuxStageBytes / 4);
          int cs = slot - R;
          if (cs < 0) cs += STAGES;
          const float* pu = ring + cs * PSTRIDE + own;  // u at plane z (landed R steps ago)
          if constexpr (!NOETA) {
#pragma unroll
            for (int k = 0; k < TYT; ++k) {
              const int a = (row0 + k) * kTX + col;
              const float4 up = lds4(pa + a);
              const float4 vv = lds4(pa + kTX * TY + a);
              const float4 et = lds4(pa + 2 * kTX * TY + a);
              const float4 uc = lds4(pu + k * BW);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float eta = get(et, e);
                const float t = fmaf(get(vv, e), pget(o[k], e),
                                     fmaf(-(1.0f - eta), get(up, e), 2.0f * get(uc, e)));
                pset(o[k], e, __fdividef(t, 1.0f + eta));  // 1 + eta in [1, 2]: 2-ulp divide
              }
            }
          } else {  // a region where eta = 0: plain leapfrog, no eta staged, no divide
#pragma unroll
            for (int k = 0; k < TYT; ++k) {
              const int a = (row0 + k) * kTX + col;
              const float4 up = lds4(pa + a);
              const float4 vv = lds4(pa + kTX * TY + a);
              const float4 uc = lds4(pu + k * BW);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                pset(o[k], e, fmaf(get(vv, e), pget(o[k], e), fmaf(2.0f, get(uc, e), -get(up, e))));
            }
          }
        }
        if constexpr (TSTORE) {
          // Stage the tile; after the next CTA barrier one thread stores it with TMA, which
          // writes only the part inside the interior (the tiles start at its origin).
          float* st = stg + stg_slot * (C::kStgPlaneBytes / 4) + row0 * kTX + col;
#pragma unroll
          for (int k = 0; k < TYT; ++k) *reinterpret_cast<float4*>(st + k * kTX) = tof4(o[k]);
          if (++stg_slot == C::kStgPlanes) stg_slot = 0;
          ++emitted;
        } else {
          float* const oz = orow + (size_t)z * plane;
#pragma unroll
          for (int k = 0; k < TYT; ++k) {
            if (row_ok[k]) {
              float* dst = oz + k * p.nx;
              if (vec_ok) {
                __stcs(reinterpret_cast<float4*>(dst), tof4(o[k]));
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (gx + e >= R && gx + e < p.nx - R) dst[e] = pget(o[k], e);
              }
            }
          }
        }
      }

      if constexpr (SEMI) {
        // Semi-stencil form, right half of the z stencil: the landed plane is the last
        // point of its R predecessors' windows; each partial sum moves one slot down.
#pragma unroll
        for (int i = 1; i < R; ++i)
#pragma unroll
          for (int k = 0; k < TYT; ++k) s[i - 1][k] = fma2x(cc[R - i], xv[k], s[i][k]);
      }

      if (j >= R && j < L - R) {
        // In-plane part of the landed plane's outputs.  Before the z filter below runs,
        // s[R] holds that plane's partial sums; the filter's FMA then carries them on
        // (they emerge R planes later).  Doing this part first measured 7 % faster than
        // after the filter: the loads issue earlier and the FMA chains overlap better.
        // In the semi-stencil form the landed plane's outputs start in the freed slot
        // s[R-1] with the centre and the left half of the z stencil, read from the R
        // planes the ring keeps behind the lead.
        P4* acc = s[SEMI ? R - 1 : R];
        if constexpr (SEMI) {
#pragma unroll
          for (int k = 0; k < TYT; ++k)
            acc[k] = P4{__fmul2_rn(cc[0], xv[k].a), __fmul2_rn(cc[0], xv[k].b)};
#pragma unroll
          for (int r = 1; r <= R; ++r) {
            int ps = slot - r;
            if (ps < 0) ps += STAGES;
            const float* q = ring + ps * PSTRIDE + own;
#pragma unroll
            for (int k = 0; k < TYT; ++k) acc[k] = fma2x(cc[r], ldp4(q + k * BW), acc[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < TYT; ++k) {
          const float* rowp = pl + own + k * BW;
          // X[0..11]: x offsets -4..7 from this thread's first column, as register pairs
          // L = X[0..3], C = X[4..7], Rt = X[8..11]; only the parts within R are loaded.
          P4 Lq, Rq;
          if constexpr (R >= 3) {
            Lq = ldp4(rowp - 4);
            Rq = ldp4(rowp + 4);
          } else if constexpr (R == 2) {
            Lq.b = *reinterpret_cast<const float2*>(rowp - 2);
            Rq.a = *reinterpret_cast<const float2*>(rowp + 4);
          } else {
            Lq.b.y = rowp[-1];
            Rq.a.x = rowp[4];
          }
          const P4& Cq = xv[k];
          auto X = [&](int i) -> float {  // scalar X[i]
            return i < 4 ? pget(Lq, i) : i < 8 ? pget(Cq, i - 4) : pget(Rq, i - 8);
          };
          auto XP = [&](int i) -> float2 {  // register pair X[i], X[i+1], i even
            return i == 0 ? Lq.a : i == 2 ? Lq.b : i == 4 ? Cq.a : i == 6 ? Cq.b : i == 8 ? Rq.a : Rq.b;
          };
#pragma unroll
          for (int r = 1; r <= R; ++r) {
            if (r % 2 == 0) {  // neighbour pairs stay register-aligned: packed
              acc[k].a = __ffma2_rn(cc[r], __fadd2_rn(XP(4 - r), XP(4 + r)), acc[k].a);
              acc[k].b = __ffma2_rn(cc[r], __fadd2_rn(XP(6 - r), XP(6 + r)), acc[k].b);
            } else {  // odd distance: pairs straddle registers, scalar
#pragma unroll
              for (int e = 0; e < 4; ++e)
                pset(acc[k], e, fmaf(cc[r].x, X(4 + e - r) + X(4 + e + r), pget(acc[k], e)));
            }
          }
        }
        // y neighbours in symmetric pairs (k-d, k+d): one add, one FMA per pair.
#pragma unroll
        for (int d = 1; d <= R; ++d) {
#pragma unroll
          for (int k = 0; k < TYT; ++k) {
            const int hm = k - d, hp = k + d;
            const P4 vm = (hm >= 0 && hm < TYT) ? xv[hm >= 0 && hm < TYT ? hm : 0] : ldp4(pl + own + hm * BW);
            const P4 vp = (hp >= 0 && hp < TYT) ? xv[hp >= 0 && hp < TYT ? hp : 0] : ldp4(pl + own + hp * BW);
            acc[k].a = __ffma2_rn(cc[d], __fadd2_rn(vm.a, vp.a), acc[k].a);
            acc[k].b = __ffma2_rn(cc[d], __fadd2_rn(vm.b, vp.b), acc[k].b);
          }
        }
      }

      if constexpr (!SEMI) {
        // z filter, transposed form: every partial sum moves one slot down.
#pragma unroll
        for (int i = 1; i < 2 * R; ++i)
#pragma unroll
          for (int k = 0; k < TYT; ++k)
            s[i - 1][k] = fma2x(cc[i < R ? R - i : i - R], xv[k], s[i][k]);
#pragma unroll
        for (int k = 0; k < TYT; ++k)
          s[2 * R - 1][k] = P4{__fmul2_rn(cc[R], xv[k].a), __fmul2_rn(cc[R], xv[k].b)};
      }

      if constexpr (DRIFT) {
        // Close the step without a CTA barrier: this warp is done with the slot of plane
        // (landed - KEEP).  The last warp to release it refills it with the plane STAGES
        // loads later, located from this warp's own progress (no shared cursor).
        const int rslot = (slot + STAGES - KEEP) % STAGES;
        ++J;
        if (++slot == STAGES) {
          slot = 0;
          phase ^= 1u;
        }
        if (__any_sync(0xffffffffu, failed)) {  // a wait of this warp ran out: leave
          failed = true;
          break;
        }
        __syncwarp();
        if (lane0 && atomicAdd(&relcnt[rslot], 1) == NWARPS - 1) {
          relcnt[rslot] = 0;  // published to the next round by the refill's arrive (release)
          int jj = j + STAGES - KEEP, it = item, L2 = L, nx0 = x0, ny0 = y0, nzs = zs, ndz = dz;
          while (jj >= L2 && it < p.nitems) {
            jj -= L2;
            it += (int)gridDim.x;
            if (it < p.nitems) item_geometry<R, TY, XO>(p, it, nx0, ny0, L2, nzs, ndz);
          }
          if (it < p.nitems) {
            const int counter = J - 1 + STAGES - KEEP;
            const uint32_t bar = base + 8u * rslot;
            lastld[rslot] = counter;
            fence_proxy_async_smem();
            if (counter != p.debug_skip) {
              mbar_arrive_expect_tx(bar, C::kPlaneBytes);
              tma_load_3d(ring_base + rslot * C::kPlaneStride, &tm_u, bar, nx0 - kHX, ny0 - R,
                          nzs + ndz * jj);
            }
          }
        }
        continue;
      }
      // Close the step.  Every KB planes (and at the end of an item) the CTA meets at a
      // barrier: every thread is then done with the slots of planes (landed - KEEP) of the
      // steps since the last barrier, and one warp (rotating) refills them.
      ++J;
      if (++slot == STAGES) {
        slot = 0;
        phase ^= 1u;
      }
      if (WAVE && ++aslot == ASTAGES) {
        aslot = 0;
        aphase ^= 1u;
      }
      if (++since < KB && j + 1 < L) continue;
      if constexpr (TSTORE) {
        fence_proxy_async_smem();  // this thread's staged tiles become visible to the TMA unit
        // The steps after this barrier stage at most KB tiles, into the slots of the group
        // issued TSTORE - 1 barriers before this one: all older groups must have read
        // theirs.  Still pending then: this barrier's group and the TSTORE - 2 before it,
        // at most (TSTORE - 1) * KB tiles right before the ones to be written.
        if (leader) bulk_wait_read<TSTORE - 2>();
      }
      const bool stop = __syncthreads_or(failed) != 0;
      if constexpr (TSTORE) {
        if (leader && !stop && emitted > 0) {
          // The planes staged since the last barrier are the last `emitted` steps'.
          for (int q = 0; q < emitted; ++q) {
            const int z = zs + dz * (j - emitted + 1 + q - R);
            int sl = stg_slot - emitted + q;
            if (sl < 0) sl += C::kStgPlanes;
            tma_store_3d(&tm_out, stg_base + sl * C::kStgPlaneBytes, x0 - R, y0 - R, z - R);
          }
          bulk_commit();
        }
        emitted = 0;
      }
      if (lane0 && !stop) {
        if (warp == pwarp) {
          fence_proxy_async_smem();
          for (int q = since; q > 0; --q) produce_u(J - q + STAGES - KEEP);
        }
        if (WAVE && warp == (pwarp + NWARPS / 2) % NWARPS) {
          fence_proxy_async_smem();
          for (int q = since; q > 0; --q) produce_aux(J - q + ASTAGES);
        }
      }
      since = 0;
      if (++pwarp == NWARPS) pwarp = 0;
      if (stop) goto drain;
    }
    if (DRIFT && failed) break;
  }
  if constexpr (DRIFT) {
    // The warps leave the loops at different times; they meet here to decide together.
    if (__syncthreads_or(failed)) goto drain;
  }
  if (TSTORE && leader) bulk_wait_all();  // the last tiles are written before the CTA leaves
  return;

drain:
  // A wait ran out: make sure none of this CTA's copies is still landing in shared
  // memory before the CTA exits (bounded as well), then leave.
  // Only the last load issued into each slot can still be outstanding.
  if (leader) {
    if (TSTORE) bulk_wait_all();
    for (int sl = 0; sl < STAGES; ++sl) {
      const int c = lastld[sl];
      if (c >= 0 && c != p.debug_skip && !mbar_wait_bounded(base + 8u * sl, (c / STAGES) & 1))
        atomicOr(p.status, kStatusDrainTimeout);
    }
    if (WAVE) {
      const int na = cur[1].issued;
      for (int c = na > ASTAGES ? na - ASTAGES : 0; c < na; ++c)
        if (!mbar_wait_bounded(base + 8u * (STAGES + c % ASTAGES), (c / ASTAGES) & 1))
          atomicOr(p.status, kStatusDrainTimeout);
    }
  }
  __syncthreads();
}

}  // namespace libstencil
