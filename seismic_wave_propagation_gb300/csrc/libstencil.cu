// libstencil C ABI: plans, argument validation, TMA descriptors, launch geometry,
// device status, and the host-buffer convenience calls.  The declarations and their
// contracts are in include/libstencil.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "libstencil.h"
#include "kernel_table.h"

using namespace libstencil;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(STENCIL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapEntry {
  const void* ptr = nullptr;
  int box_w = 0, box_h = 0;
  int view = 0;  // 0: the whole grid; 1: its interior (points at least R from every face)
  uint64_t stamp = 0;
  CUtensorMap map;
};

constexpr int kMapCache = 16;

}  // namespace

struct stencil_plan {
  int64_t nx, ny, nz;
  int radius;
  float c[STENCIL_MAX_RADIUS + 1];
  int device;
  int num_sms;
  // [0] apply, [1] wave, [2] wave without eta (inner region of wave_step_pml), [3] semi
  // apply, [4] two sweeps in one pass (radius 1 only; fn null otherwise)
  KernelDesc kd[5];
  int occupancy[5];    // CTAs per SM
  StarParams params[5];
  int grid[5];
  unsigned* d_status;  // 4 words
  MapEntry maps[kMapCache];
  uint64_t clock;
  float* work;         // host-API workspace
  size_t work_floats;
  int debug_mode;
  // Cached CUDA graph of the last multi-launch loop (stencil_sweeps / wave_steps).
  cudaGraphExec_t graph;
  uint64_t graph_key[8];
  // Streams and events of the slab-pipelined host-buffer sweep (created on first use).
  cudaStream_t pipe[3];  // copies in, compute, copies out
  cudaEvent_t ev[2 * 32 + 2];
  bool pipe_ready;
  int pipe_slabs;        // slabs of the last pipelined call (0: none yet)
  stencil_plan* eta_plan;  // radius-1 plan of the same grid for wave_eta_stencil (on first use)
  // The band launch of wave_step_pml runs on `side`, beside the inner region's launch.
  cudaStream_t side;
  cudaEvent_t side_fork, side_join;
  // Geometry of the last band width (wave_step_pml): inner region and band launches.
  int64_t reg_pml;         // -1: none yet
  int reg_kind;            // 2: inner and band; 1: no inner region (one full launch)
  StarParams reg_inner, reg_band;
  int reg_inner_grid, reg_band_grid;
  // Sweep path of stencil_apply and the sweep loops: STENCIL_PATH_AUTO (chosen by grid
  // size), _STAGED or _DIRECT; `direct` is the resolved choice.
  int sweep_path;
  bool direct;
  int direct_occupancy;  // blocks of the direct kernel per SM
};

namespace {

int64_t npoints(const stencil_plan* p) { return p->nx * p->ny * p->nz; }

bool interior_empty(const stencil_plan* p) {
  const int64_t m = 2 * (int64_t)p->radius + 1;
  return p->nx < m || p->ny < m || p->nz < m;
}

// The z-chunk schedule for `nzi` output planes of x-y tiles of height tile_y: the number
// of chunks per tile column, minimising the per-CTA step count of the round-robin
// schedule over `slots` CTA slots (a filling step costs about a third of a computing one);
// light sweeps instead take the fewest chunks that occupy every SM.
//
// Only one chunk count per round count can win: with k rounds, n_k = floor(k * slots /
// ntiles) chunks (at least 1, at most nzi) is the most that still fit, and any smaller n
// with k rounds has as many rounds, no fewer steps per item and fewer busy slots.  The
// scan therefore visits round counts, not chunk counts, and its cost does not grow with
// nz (at most kMaxRounds candidates).
struct Schedule {
  int ntx, ntiles, nchunks, nitems, grid;
};

constexpr int64_t kMaxRounds = 1 << 14;

// Tiles along x and y: they cover x from 0 (masked stores) or from the interior origin R
// (TMA stores), and y from R.
void tile_grid(int64_t nx, int64_t ny, int R, int tile_y, bool interior_tiles, int& ntx, int& nty) {
  const int64_t xext = interior_tiles ? nx - 2 * R : nx;
  ntx = (int)((xext + kTX - 1) / kTX);
  nty = (int)((ny - 2 * R + tile_y - 1) / tile_y);
}

// Chunks per tile column for `ntiles` tiles and `nzi` output planes (the scan above).
int64_t choose_chunks(int64_t ntiles, int nzi, int R, int kind, int num_sms, int occupancy) {
  const int64_t slots = (int64_t)num_sms * std::max(1, occupancy);
  // Cost of n chunks: rounds of the round-robin schedule x steps per item; and the share
  // of the GPU's CTA slots the schedule keeps busy (a partly filled round idles the rest).
  auto plan_n = [&](int64_t n, double& cost, double& busy) {
    const int64_t items = ntiles * n;
    const int64_t g = std::min<int64_t>(items, slots);
    const int64_t rounds = (items + g - 1) / g;
    cost = (double)rounds * ((double)((nzi + n - 1) / n) + 0.35 * 2 * R);
    busy = (double)items / (double)(rounds * slots);
  };
  const int64_t max_n = std::min<int64_t>(nzi, ((int64_t)1 << 30) / ntiles);
  auto candidate = [&](int64_t k) {
    return std::min<int64_t>(max_n, std::max<int64_t>(1, k * slots / ntiles));
  };
  double best = 1e300, cost, busy;
  for (int64_t k = 1, last = 0; k <= kMaxRounds; ++k) {
    const int64_t n = candidate(k);
    if (n == last) continue;
    last = n;
    plan_n(n, cost, busy);
    best = std::min(best, cost);
    if (n == max_n) break;
  }
  // Among near-ties (within 0.5 %), take the fullest schedule: at 1536 x 1536 x 256,
  // R = 4, 1 and 5 chunks cost the same, and 5 (a 95 % full last round instead of 79 %)
  // measured 5 % faster.
  int64_t best_n = 1;
  double best_busy = -1.0;
  for (int64_t k = 1, last = 0; k <= kMaxRounds; ++k) {
    const int64_t n = candidate(k);
    if (n == last) continue;
    last = n;
    plan_n(n, cost, busy);
    if (cost <= best * 1.005 && busy > best_busy + 1e-12) {
      best_busy = busy;
      best_n = n;
    }
    if (n == max_n) break;
  }
  if ((kind == 0 || kind == 3) && R <= 2) {
    // Light sweeps are bound by memory traffic, not by the busiest SM: the fewest chunks
    // that still give every SM a CTA keep the fewest z-fronts in flight and the fewest
    // refilled planes (measured at 512^3, R = 1: 2 chunks 5.7 TB/s, 7 chunks 4.9 TB/s).
    best_n = std::min<int64_t>(nzi, ((int64_t)num_sms + ntiles - 1) / ntiles);
  }
  return best_n;
}

Schedule schedule(int64_t nx, int64_t ny, int R, int tile_y, int kind, int num_sms, int occupancy,
                  int nzi, bool interior_tiles) {
  Schedule sc{};
  int nty;
  tile_grid(nx, ny, R, tile_y, interior_tiles, sc.ntx, nty);
  sc.ntiles = sc.ntx * nty;
  const int64_t slots = (int64_t)num_sms * std::max(1, occupancy);
  sc.nchunks = (int)choose_chunks(sc.ntiles, nzi, R, kind, num_sms, occupancy);
  sc.nitems = (int)((int64_t)sc.ntiles * sc.nchunks);
  sc.grid = (int)std::min<int64_t>(sc.nitems, slots);
  return sc;
}

// A rectangle of tiles [tx0, tx0 + ntx) x [ty0, ty0 + nty) and the output planes
// [z0, z0 + nzi).
struct Region {
  int tx0, ty0, ntx, nty, z0, nzi;
};

// Several regions in one launch on `slots` CTAs: every box is cut into chunks of about T
// output planes (thin boxes stay whole), the boxes with the longest items first, and T is
// the one whose round-robin deal gives the smallest busiest CTA (a filling step counted as
// 0.35 of a computing one).  Returns that busiest CTA's load in steps.
double plan_regions(Region* rg, int nr, int R, int64_t slots, Box* box, int& nitems) {
  std::stable_sort(rg, rg + nr, [](const Region& a, const Region& b) { return a.nzi > b.nzi; });
  int zmax = 1;
  for (int b = 0; b < nr; ++b) zmax = std::max(zmax, rg[b].nzi);
  std::vector<double> load((size_t)std::max<int64_t>(1, slots));
  double best = 1e300;
  int best_t = zmax;
  for (int n = 1; n <= std::min(zmax, 64); ++n) {
    const int T = (zmax + n - 1) / n;
    std::fill(load.begin(), load.end(), 0.0);
    int64_t item = 0;
    for (int b = 0; b < nr; ++b) {
      const int c = std::min(rg[b].nzi, std::max(1, (rg[b].nzi + T / 2) / T));
      const double len = (double)((rg[b].nzi + c - 1) / c) + 0.35 * 2 * R;
      const int64_t cnt = (int64_t)rg[b].ntx * rg[b].nty * c;
      for (int64_t i = 0; i < cnt; ++i, ++item) load[(size_t)(item % slots)] += len;
    }
    const double worst = *std::max_element(load.begin(), load.end());
    if (worst < best * 0.999) {
      best = worst;
      best_t = T;
    }
  }
  nitems = 0;
  for (int b = 0; b < nr; ++b) {
    const int c = std::min(rg[b].nzi, std::max(1, (rg[b].nzi + best_t / 2) / best_t));
    box[b] = Box{rg[b].tx0, rg[b].ty0, rg[b].ntx, rg[b].ntx * rg[b].nty, rg[b].z0, rg[b].nzi, c, nitems};
    nitems += box[b].ntiles * c;
  }
  return best;
}

// Launch geometry for the output planes [R + zoff, R + zoff + nzi) of the grid.
void geometry(const stencil_plan* p, int kind, int zoff, int nzi, StarParams& sp, int& grid) {
  const KernelDesc& kd = p->kd[kind];
  const int R = p->radius;
  std::memset(&sp, 0, sizeof sp);
  sp.nx = (int)p->nx;
  sp.ny = (int)p->ny;
  sp.nz = (int)p->nz;
  for (int r = 0; r <= 4; ++r) sp.c[r] = r <= R ? p->c[r] : 0.0f;
  sp.status = p->d_status;
  sp.debug_skip = -1;
  if (interior_empty(p) || nzi <= 0) {
    grid = 0;
    return;
  }
  const Schedule sc =
      schedule(p->nx, p->ny, R, kd.tile_y, kind, p->num_sms, p->occupancy[kind], nzi, kd.tstore);
  sp.nboxes = 1;
  sp.box[0] = Box{0, 0, sc.ntx, sc.ntiles, R + zoff, nzi, sc.nchunks, 0};
  sp.nitems = sc.nitems;
  grid = sc.grid;
}

// Launch geometry for a list of regions (at most kMaxBoxes, none empty) on `slots` CTAs.
// One region is chunked by the scan over round counts, several by plan_regions.
void geometry_regions(const stencil_plan* p, int kind, Region* rg, int nr, int64_t slots,
                      StarParams& sp, int& grid) {
  geometry(p, kind, 0, 0, sp, grid);  // fields, coefficients, status; no work yet
  if (nr == 1) {
    const int ntiles = rg[0].ntx * rg[0].nty;
    const int n = (int)choose_chunks(ntiles, rg[0].nzi, p->radius, kind, (int)slots, 1);
    sp.nboxes = 1;
    sp.box[0] = Box{rg[0].tx0, rg[0].ty0, rg[0].ntx, ntiles, rg[0].z0, rg[0].nzi, n, 0};
    sp.nitems = ntiles * n;
  } else {
    sp.nboxes = nr;
    plan_regions(rg, nr, p->radius, slots, sp.box, sp.nitems);
  }
  grid = (int)std::min<int64_t>(sp.nitems, slots);
}

void plan_geometry(stencil_plan* p, int kind) {
  geometry(p, kind, 0, (int)(p->nz - 2 * p->radius), p->params[kind], p->grid[kind]);
}

int check_device(const stencil_plan* p) {
  int d = -1;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (d != p->device)
    return fail(STENCIL_ERR_ARG, "current device %d is not the plan's device %d", d, p->device);
  return STENCIL_OK;
}

int check_field(const stencil_plan* p, const void* ptr, const char* name) {
  if (!ptr) return fail(STENCIL_ERR_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(ptr) & 15u)
    return fail(STENCIL_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(STENCIL_ERR_ARG, "%s is not a CUDA pointer (%s)", name, cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(STENCIL_ERR_ARG, "%s is not device memory", name);
  if (a.device != p->device)
    return fail(STENCIL_ERR_ARG, "%s lives on device %d, the plan on device %d", name, a.device,
                p->device);
  return STENCIL_OK;
}

bool overlap(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

// TMA descriptor for a field pointer and box shape (cached per plan).  view 1 maps the
// interior only: its origin is the point (R, R, R), so a box stored through it never writes
// the shell (the TMA unit drops the parts of a box outside the tensor).
int get_map(stencil_plan* p, const void* ptr, int box_w, int box_h, const CUtensorMap** out,
            int view = 0) {
  MapEntry* victim = &p->maps[0];
  for (MapEntry& m : p->maps) {
    if (m.ptr == ptr && m.box_w == box_w && m.box_h == box_h && m.view == view) {
      m.stamp = ++p->clock;
      *out = &m.map;
      return STENCIL_OK;
    }
    if (m.stamp < victim->stamp) victim = &m;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return fail(STENCIL_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const int64_t e = view ? 2 * p->radius : 0;
  const cuuint64_t dims[3] = {(cuuint64_t)(p->nx - e), (cuuint64_t)(p->ny - e), (cuuint64_t)(p->nz - e)};
  const cuuint64_t strides[2] = {(cuuint64_t)p->nx * 4, (cuuint64_t)(p->nx * p->ny) * 4};
  const cuuint32_t box[3] = {(cuuint32_t)box_w, (cuuint32_t)box_h, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const int64_t org = view ? p->radius * (1 + p->nx + p->nx * p->ny) : 0;  // floats to (R, R, R)
  void* gbase = const_cast<float*>(static_cast<const float*>(ptr)) + org;
  if (reinterpret_cast<uintptr_t>(gbase) & 15u)
    return fail(STENCIL_ERR_ALIGNMENT, "interior origin of the output is not 16-byte aligned");
  CUresult r = enc(&victim->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, gbase, dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    victim->ptr = nullptr;
    victim->stamp = 0;
    return fail(STENCIL_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  }
  victim->ptr = ptr;
  victim->box_w = box_w;
  victim->box_h = box_h;
  victim->view = view;
  victim->stamp = ++p->clock;
  *out = &victim->map;
  return STENCIL_OK;
}

// Grids up to this many points (per radius) sweep faster with the direct-load kernel than
// with the staged one: there the launch and pipeline-filling latency of the staged kernel
// outweighs its saving in loads.  Measured on GB300, one sweep launched after another, on
// cubes: radius 1 direct faster through 448^3 (136 against 149 us), slower at 512^3;
// radius 2 through 224^3, slower at 256^3; radius 3 through 160^3, slower at 192^3;
// radius 4 through 144^3 (12.3 against 14.4 us), slower at 160^3.
constexpr int64_t kDirectMaxPoints[STENCIL_MAX_RADIUS + 1] = {0, 100000000, 12000000, 5000000, 3500000};
// Radius-1 loops on the automatic path: from this many points a two-sweep pass of the
// staged kernel beats two direct sweeps (GB300, chained in a graph, per sweep: 192^3 10.81
// against 10.63 us, 224^3 16.1 against 19.1, 256^3 20.9 against 27.1).
constexpr int64_t kPairMinPoints = 8000000;

bool resolve_direct(const stencil_plan* p) {
  if (p->sweep_path == STENCIL_PATH_DIRECT) return true;
  if (p->sweep_path == STENCIL_PATH_STAGED) return false;
  return npoints(p) <= kDirectMaxPoints[p->radius];
}

// Geometry of a direct-kernel sweep over output planes [R + zoff, R + zoff + nzi).
DirectParams direct_params(const stencil_plan* p, const float* in, float* out, int zoff, int nzi,
                           int64_t& blocks) {
  const int R = p->radius;
  DirectParams d{};
  d.in = in;
  d.out = out;
  d.nx = (int)p->nx;
  d.ny = (int)p->ny;
  d.z0 = R + zoff;
  d.q0 = R >> 2;                                   // first float4 column with x >= R
  d.nq = (int)(((p->nx - R - 1) >> 2) + 1) - d.q0;  // through the column with x = nx - R - 1
  d.nyi = (int)(p->ny - 2 * R);
  d.total = interior_empty(p) || nzi <= 0 ? 0 : (int64_t)d.nq * d.nyi * nzi;
  for (int r = 0; r <= STENCIL_MAX_RADIUS; ++r) d.c[r] = p->c[r];
  blocks = (d.total + kDirectThreads - 1) / kDirectThreads;
  return d;
}

int launch_direct_sweep(stencil_plan* p, const float* in, float* out, cudaStream_t stream, int zoff,
                        int nzi) {
  if (nzi < 0) nzi = (int)(p->nz - 2 * p->radius);
  int64_t blocks = 0;
  const DirectParams d = direct_params(p, in, out, zoff, nzi, blocks);
  if (blocks == 0) return STENCIL_OK;  // empty interior: nothing to do
  if (blocks > INT32_MAX) return fail(STENCIL_ERR_ARG, "grid too large for the direct sweep");
  cudaError_t e = launch_direct(p->radius, dim3((unsigned)blocks), stream, d);
  return e == cudaSuccess ? STENCIL_OK : cuda_fail(e, "kernel launch");
}

// Launch one sweep (kind 0, 3) or wave step (1; 2 = without eta).  nzi >= 0 restricts it
// to the output planes [R + zoff, R + zoff + nzi); `geo` (with `geo_grid` CTAs) gives the
// work of the launch explicitly.
int launch(stencil_plan* p, int kind, const float* u, const float* uprev, const float* v2dt2,
           const float* eta, float* out, cudaStream_t stream, int zoff = 0, int nzi = -1,
           const StarParams* geo = nullptr, int geo_grid = 0) {
  if (kind == 0 && p->direct && !geo) return launch_direct_sweep(p, u, out, stream, zoff, nzi);
  StarParams sp = geo ? *geo : p->params[kind];
  int grid = geo ? geo_grid : p->grid[kind];
  if (!geo && nzi >= 0) geometry(p, kind, zoff, nzi, sp, grid);
  if (grid == 0) return STENCIL_OK;  // empty interior: nothing to do
  const KernelDesc& kd = p->kd[kind];
  const CUtensorMap *mu, *mp = nullptr, *mv = nullptr, *me = nullptr;
  int rc = get_map(p, u, kd.box_w, kd.box_h, &mu);
  if (rc) return rc;
  if (kind == 1 || kind == 2) {
    if ((rc = get_map(p, uprev, kTX, kd.tile_y, &mp))) return rc;
    if ((rc = get_map(p, v2dt2, kTX, kd.tile_y, &mv))) return rc;
    if ((rc = get_map(p, eta, kTX, kd.tile_y, &me))) return rc;
  } else {
    mp = mv = me = mu;
  }
  const CUtensorMap* mo = mu;
  if (kd.tstore && (rc = get_map(p, out, kTX, kd.tile_y, &mo, 1))) return rc;
  sp.out = out;
  sp.debug_skip = p->debug_mode == 1 ? 0 : -1;  // every CTA has a load 0
  // Copy the descriptors: the cache may evict entries while the launch is pending.
  const CUtensorMap a = *mu, b = *mp, c = *mv, d = *me, o = *mo;
  cudaError_t e = kd.launch(dim3(grid), stream, a, b, c, d, o, sp);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return STENCIL_OK;
}

int ensure_work(stencil_plan* p, size_t floats) {
  if (p->work_floats >= floats) return STENCIL_OK;
  if (p->work) cudaFree(p->work);
  p->work = nullptr;
  p->work_floats = 0;
  cudaError_t e = cudaMalloc(&p->work, floats * sizeof(float));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
  p->work_floats = floats;
  return STENCIL_OK;
}

}  // namespace

namespace {

// Enqueue `body` (a sequence of launches on `s`) directly, or as a CUDA graph captured
// once per distinct key and replayed afterwards.
template <class Body>
int run_loop(stencil_plan* p, const uint64_t key[8], bool use_graph, cudaStream_t s, Body body) {
  if (!use_graph) return body(s);
  if (!p->graph || std::memcmp(key, p->graph_key, sizeof p->graph_key) != 0) {
    if (p->graph) {
      cudaGraphExecDestroy(p->graph);
      p->graph = nullptr;
    }
    cudaStream_t cap;
    cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "capture stream");
    e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    int rc = STENCIL_OK;
    if (e == cudaSuccess) rc = body(cap);
    cudaGraph_t g = nullptr;
    const cudaError_t e2 = cudaStreamEndCapture(cap, &g);
    cudaStreamDestroy(cap);
    if (e != cudaSuccess) return cuda_fail(e, "begin capture");
    if (rc) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    if (e2 != cudaSuccess) return cuda_fail(e2, "end capture");
    e = cudaGraphInstantiate(&p->graph, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      p->graph = nullptr;
      return cuda_fail(e, "graph instantiate");
    }
    std::memcpy(p->graph_key, key, sizeof p->graph_key);
  }
  cudaError_t e = cudaGraphLaunch(p->graph, s);
  return e == cudaSuccess ? STENCIL_OK : cuda_fail(e, "graph launch");
}

}  // namespace

namespace {

// One sweep from host to host, pipelined over z-slabs on three streams so that the copy
// in of later slabs, the sweep of the current one and the copy out of earlier ones
// overlap.  Slab k computes output planes [z_k, z_k+1); it needs input planes up to
// z_k+1 + R - 1, which the copy-in chunks [p_k, p_k+1) with p_k = z_k + R deliver in
// order.  Its output chunk [o_k, o_k+1) (o_k = z_k, widened to the grid's first and last
// planes at the ends) is first filled from the input (the shell), then swept, then
// copied out.
int apply_host_pipelined(stencil_plan* p, const float* in_host, float* out_host, float* a, float* b,
                         cudaStream_t user) {
  const int R = p->radius;
  const int nz = (int)p->nz;
  const int nzi = nz - 2 * R;
  const size_t plane = (size_t)p->nx * p->ny;
  cudaError_t e = cudaSuccess;
  if (!p->pipe_ready) {
    for (cudaStream_t& q : p->pipe)
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking);
    for (cudaEvent_t& v : p->ev)  // timing events: stencil_plan_host_phases reads them
      if (e == cudaSuccess) e = cudaEventCreate(&v);
    if (e != cudaSuccess) return cuda_fail(e, "pipeline streams");
    p->pipe_ready = true;
  }
  const int K = std::max(1, std::min(32, nzi / 32));
  auto zk = [&](int k) { return R + (int)(((int64_t)k * nzi) / K); };
  auto pk = [&](int k) { return k == 0 ? 0 : k == K ? nz : zk(k) + R; };
  auto ok = [&](int k) { return k == 0 ? 0 : k == K ? nz : zk(k); };
  cudaStream_t hin = p->pipe[0], comp = p->pipe[1], hout = p->pipe[2];
  cudaEvent_t start = p->ev[2 * 32], done = p->ev[2 * 32 + 1];
  e = cudaEventRecord(start, user);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hin, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hout, start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "pipeline start");
  for (int k = 0; k < K; ++k) {
    cudaEvent_t landed = p->ev[k], swept = p->ev[32 + k];
    const size_t i0 = (size_t)pk(k) * plane, i1 = (size_t)pk(k + 1) * plane;
    const size_t o0 = (size_t)ok(k) * plane, o1 = (size_t)ok(k + 1) * plane;
    e = cudaMemcpyAsync(a + i0, in_host + i0, (i1 - i0) * 4, cudaMemcpyHostToDevice, hin);
    if (e == cudaSuccess) e = cudaEventRecord(landed, hin);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, landed, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b + o0, a + o0, (o1 - o0) * 4, cudaMemcpyDeviceToDevice, comp);
    if (e != cudaSuccess) return cuda_fail(e, "pipelined copy in");
    const int rc = launch(p, 0, a, nullptr, nullptr, nullptr, b, comp, zk(k) - R, zk(k + 1) - zk(k));
    if (rc) return rc;
    e = cudaEventRecord(swept, comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hout, swept, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_host + o0, b + o0, (o1 - o0) * 4, cudaMemcpyDeviceToHost, hout);
    if (e != cudaSuccess) return cuda_fail(e, "pipelined copy out");
  }
  e = cudaEventRecord(done, hout);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(user, done, 0);
  if (e != cudaSuccess) return cuda_fail(e, "pipeline end");
  p->pipe_slabs = K;
  return stencil_plan_status(p, user);
}

// wave_step_pml as two launches: the inner region, where eta is zero, with the kernel that
// stages no eta and never divides; and the band along the faces (at most six boxes) with
// the full update, launched after it on the side stream, so that the band's items take
// the SMs the inner launch frees.  The inner region is every tile lying wholly at least
// `pml` points from the x and y faces, over the output planes at least `pml` from the z
// faces.  The geometry of both is kept for the last band width.
void plan_regions_for(stencil_plan* p, int64_t pml) {
  const int R = p->radius;
  p->reg_pml = pml;
  p->reg_kind = 1;
  if (interior_empty(p)) return;
  const KernelDesc& kd = p->kd[1];
  const int xo = kd.tstore ? R : 0;
  int ntx, nty;
  tile_grid(p->nx, p->ny, R, kd.tile_y, kd.tstore, ntx, nty);
  const int64_t TY = kd.tile_y;
  const int bx0 = (int)std::max<int64_t>(0, (pml - xo + kTX - 1) / kTX);
  const int bx1 = (int)std::min<int64_t>(ntx, p->nx - pml - xo >= 0 ? (p->nx - pml - xo) / kTX : 0);
  const int by0 = (int)std::max<int64_t>(0, (pml - R + TY - 1) / TY);
  const int by1 = (int)std::min<int64_t>(nty, p->ny - pml - R >= 0 ? (p->ny - pml - R) / TY : 0);
  const int z0 = (int)std::max<int64_t>(R, pml), z1 = (int)std::min<int64_t>(p->nz - R, p->nz - pml);
  if (bx0 >= bx1 || by0 >= by1 || z0 >= z1) return;  // no inner region: the full update everywhere
  Region band[kMaxBoxes];
  int nb = 0;
  const int zall0 = R, zall1 = (int)p->nz - R;
  if (z0 > zall0) band[nb++] = Region{0, 0, ntx, nty, zall0, z0 - zall0};
  if (z1 < zall1) band[nb++] = Region{0, 0, ntx, nty, z1, zall1 - z1};
  if (by0 > 0) band[nb++] = Region{0, 0, ntx, by0, z0, z1 - z0};
  if (by1 < nty) band[nb++] = Region{0, by1, ntx, nty - by1, z0, z1 - z0};
  if (bx0 > 0) band[nb++] = Region{0, by0, bx0, by1 - by0, z0, z1 - z0};
  if (bx1 < ntx) band[nb++] = Region{bx1, by0, ntx - bx1, by1 - by0, z0, z1 - z0};
  Region inner{bx0, by0, bx1 - bx0, by1 - by0, z0, z1 - z0};
  // Both launches are planned on all CTA slots and run side by side; the band's items
  // take the slots the inner launch leaves or frees.  (Dividing the slots between them in
  // proportion to their work, or running the band after the inner region, measured slower.)
  // Split only where the inner region holds at least 0.6 of the work: its points cost 0.84
  // of the band's (640^3: 0.654 ms for a step with no eta anywhere, 0.78 ms with eta), and
  // a thicker band of 64-wide tiles costs more in packing than that saves.  Measured on
  // GB300 (16-point band unless noted), split against one launch: 640^3 (inner share 0.71)
  // -6 %, 640^3 with a 32-point band (0.64) -3 %, 512^3 (0.65) -2 %, 384^3 (0.55) +8 %.
  const double all = (double)ntx * nty * (zall1 - zall0);
  if ((double)inner.ntx * inner.nty * inner.nzi < 0.6 * all) return;
  const int64_t slots = (int64_t)p->num_sms * std::max(1, std::min(p->occupancy[1], p->occupancy[2]));
  geometry_regions(p, 2, &inner, 1, slots, p->reg_inner, p->reg_inner_grid);
  p->reg_band_grid = 0;
  if (nb > 0) geometry_regions(p, 1, band, nb, slots, p->reg_band, p->reg_band_grid);
  p->reg_kind = 2;
}

int wave_step_regions(stencil_plan* p, const float* u_prev, const float* u, float* u_next,
                      const float* v2dt2, const float* eta, int64_t pml, cudaStream_t s) {
  if (p->reg_pml != pml) plan_regions_for(p, pml);
  if (p->reg_kind == 1) return launch(p, 1, u, u_prev, v2dt2, eta, u_next, s);
  const bool band = p->reg_band_grid > 0;
  cudaError_t e = cudaSuccess;
  if (band) {  // the band may start once the work before this step is done, not the inner part
    e = cudaEventRecord(p->side_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->side_fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "band fork");
  }
  int rc = launch(p, 2, u, u_prev, v2dt2, eta, u_next, s, 0, -1, &p->reg_inner, p->reg_inner_grid);
  if (rc || !band) return rc;
  if ((rc = launch(p, 1, u, u_prev, v2dt2, eta, u_next, p->side, 0, -1, &p->reg_band, p->reg_band_grid)))
    return rc;
  e = cudaEventRecord(p->side_join, p->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->side_join, 0);
  return e == cudaSuccess ? STENCIL_OK : cuda_fail(e, "band join");
}

// `n` ping-pong sweeps x -> y -> x ... on stream s.  Where the plan has the two-sweep
// kernel (radius 1), most of them run in pairs, one pass per pair, on the staged path and,
// on the automatic path, from kPairMinPoints up (below, two direct sweeps are faster);
// the number of such passes is kept even so that the result lands where n single sweeps
// would leave it (x for even n, y for odd n): 2*floor(n/4) passes, then the rest one by
// one on the plan's sweep path.
bool loop_pairs(const stencil_plan* p) {
  if (!p->kd[4].fn || p->sweep_path == STENCIL_PATH_DIRECT) return false;
  return p->sweep_path == STENCIL_PATH_STAGED || npoints(p) >= kPairMinPoints;
}

int ping_pong(stencil_plan* p, float* x, float* y, int n, cudaStream_t s) {
  const int pairs = loop_pairs(p) ? 2 * (n / 4) : 0;
  for (int i = 0; i < pairs; ++i) {
    const int r = launch(p, 4, x, nullptr, nullptr, nullptr, y, s);
    if (r) return r;
    std::swap(x, y);
  }
  for (int i = 2 * pairs; i < n; ++i) {
    const int r = launch(p, 0, x, nullptr, nullptr, nullptr, y, s);
    if (r) return r;
    std::swap(x, y);
  }
  return STENCIL_OK;
}

}  // namespace

extern "C" {

const char* stencil_last_error(void) { return g_err; }

const char* stencil_version(void) { return "libstencil 0.1 (sm_103a)"; }

stencil_plan* stencil_plan_create(int64_t nx, int64_t ny, int64_t nz, int radius,
                                  const float* coeffs) {
  g_err[0] = 0;
  if (radius < 1 || radius > STENCIL_MAX_RADIUS) {
    fail(STENCIL_ERR_ARG, "radius %d outside [1, %d]", radius, STENCIL_MAX_RADIUS);
    return nullptr;
  }
  if (!coeffs) {
    fail(STENCIL_ERR_ARG, "coeffs is NULL");
    return nullptr;
  }
  if (nx < 1 || ny < 1 || nz < 1 || nx > (1 << 30) || ny > (1 << 30) || nz > (1 << 30) ||
      nx * ny > ((int64_t)1 << 40) || nx * ny * nz > ((int64_t)1 << 40)) {
    fail(STENCIL_ERR_ARG, "grid %lld x %lld x %lld out of range", (long long)nx, (long long)ny,
         (long long)nz);
    return nullptr;
  }
  if (nx % 4) {
    fail(STENCIL_ERR_ALIGNMENT, "nx = %lld is not a multiple of 4", (long long)nx);
    return nullptr;
  }
  stencil_plan* p = new stencil_plan();
  p->reg_pml = -1;
  p->nx = nx;
  p->ny = ny;
  p->nz = nz;
  p->radius = radius;
  for (int r = 0; r <= STENCIL_MAX_RADIUS; ++r) p->c[r] = r <= radius ? coeffs[r] : 0.0f;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e == cudaSuccess) e = cudaMalloc(&p->d_status, 4 * sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(p->d_status, 0, 4 * sizeof(unsigned));
  // The side stream of wave_step_pml's band launch (created here, not under a capture).
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->side_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->side_join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cuda_fail(e, "plan setup");
    stencil_plan_destroy(p);
    return nullptr;
  }
  p->kd[0] = apply_kernel_desc(radius, nx, ny);
  p->kd[1] = wave_kernel_desc(radius, false);
  p->kd[2] = wave_kernel_desc(radius, true);
  p->kd[3] = semi_kernel_desc(radius);
  p->kd[4] = apply2_kernel_desc(radius);
  for (int k = 0; k < 5; ++k) {
    if (!p->kd[k].fn) continue;  // not built for this radius
    e = cudaFuncSetAttribute(p->kd[k].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p->kd[k].smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p->occupancy[k], p->kd[k].fn,
                                                        p->kd[k].threads, p->kd[k].smem);
    if (e != cudaSuccess || p->occupancy[k] < 1) {
      if (e == cudaSuccess) fail(STENCIL_ERR_CUDA, "kernel cannot be resident (occupancy 0)");
      else cuda_fail(e, "kernel attributes");
      stencil_plan_destroy(p);
      return nullptr;
    }
    plan_geometry(p, k);
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&p->direct_occupancy, direct_kernel_fn(radius),
                                                    kDirectThreads, 0);
  if (e != cudaSuccess) {
    cuda_fail(e, "kernel attributes");
    stencil_plan_destroy(p);
    return nullptr;
  }
  p->sweep_path = STENCIL_PATH_AUTO;
  p->direct = resolve_direct(p);
  return p;
}

void stencil_plan_destroy(stencil_plan* p) {
  if (!p) return;
  if (p->side) cudaStreamDestroy(p->side);
  if (p->side_fork) cudaEventDestroy(p->side_fork);
  if (p->side_join) cudaEventDestroy(p->side_join);
  if (p->eta_plan) stencil_plan_destroy(p->eta_plan);
  if (p->graph) cudaGraphExecDestroy(p->graph);
  if (p->pipe_ready) {
    for (cudaStream_t q : p->pipe) cudaStreamDestroy(q);
    for (cudaEvent_t v : p->ev) cudaEventDestroy(v);
  }
  if (p->d_status) cudaFree(p->d_status);
  if (p->work) cudaFree(p->work);
  delete p;
}

int stencil_apply(stencil_plan* p, const float* in, float* out, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, in, "in")) || (rc = check_field(p, out, "out"))) return rc;
  if (overlap(in, out, (size_t)npoints(p) * 4)) return fail(STENCIL_ERR_ALIAS, "in and out overlap");
  return launch(p, 0, in, nullptr, nullptr, nullptr, out, static_cast<cudaStream_t>(stream));
}

int stencil_apply2(stencil_plan* p, const float* in, float* out, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (!p->kd[4].fn) return fail(STENCIL_ERR_ARG, "two sweeps per pass are built for radius 1, not %d", p->radius);
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, in, "in")) || (rc = check_field(p, out, "out"))) return rc;
  if (overlap(in, out, (size_t)npoints(p) * 4)) return fail(STENCIL_ERR_ALIAS, "in and out overlap");
  return launch(p, 4, in, nullptr, nullptr, nullptr, out, static_cast<cudaStream_t>(stream));
}

int stencil_apply_semi(stencil_plan* p, const float* in, float* out, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, in, "in")) || (rc = check_field(p, out, "out"))) return rc;
  if (overlap(in, out, (size_t)npoints(p) * 4)) return fail(STENCIL_ERR_ALIAS, "in and out overlap");
  return launch(p, 3, in, nullptr, nullptr, nullptr, out, static_cast<cudaStream_t>(stream));
}

int wave_step(stencil_plan* p, const float* u_prev, const float* u, float* u_next,
              const float* v2dt2, const float* eta, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, u_prev, "u_prev")) || (rc = check_field(p, u, "u")) ||
      (rc = check_field(p, u_next, "u_next")) || (rc = check_field(p, v2dt2, "v2dt2")) ||
      (rc = check_field(p, eta, "eta")))
    return rc;
  const size_t bytes = (size_t)npoints(p) * 4;
  if (overlap(u_next, u, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps u");
  if (overlap(u_next, v2dt2, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps v2dt2");
  if (overlap(u_next, eta, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps eta");
  if (u_next != u_prev && overlap(u_next, u_prev, bytes))
    return fail(STENCIL_ERR_ALIAS, "u_next partially overlaps u_prev");
  return launch(p, 1, u, u_prev, v2dt2, eta, u_next, static_cast<cudaStream_t>(stream));
}

int wave_step_pml(stencil_plan* p, const float* u_prev, const float* u, float* u_next,
                  const float* v2dt2, const float* eta, int64_t pml_width, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (pml_width < 0) return fail(STENCIL_ERR_ARG, "pml_width < 0");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, u_prev, "u_prev")) || (rc = check_field(p, u, "u")) ||
      (rc = check_field(p, u_next, "u_next")) || (rc = check_field(p, v2dt2, "v2dt2")) ||
      (rc = check_field(p, eta, "eta")))
    return rc;
  const size_t bytes = (size_t)npoints(p) * 4;
  if (overlap(u_next, u, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps u");
  if (overlap(u_next, v2dt2, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps v2dt2");
  if (overlap(u_next, eta, bytes)) return fail(STENCIL_ERR_ALIAS, "u_next overlaps eta");
  if (u_next != u_prev && overlap(u_next, u_prev, bytes))
    return fail(STENCIL_ERR_ALIAS, "u_next partially overlaps u_prev");
  return wave_step_regions(p, u_prev, u, u_next, v2dt2, eta, std::min<int64_t>(pml_width, 1 << 30),
                           static_cast<cudaStream_t>(stream));
}

int wave_eta_stencil(stencil_plan* p, const float* eta, float* eta_eff, float e0, float e1, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, eta, "eta")) || (rc = check_field(p, eta_eff, "eta_eff"))) return rc;
  const size_t bytes = (size_t)npoints(p) * 4;
  if (overlap(eta, eta_eff, bytes)) return fail(STENCIL_ERR_ALIAS, "eta and eta_eff overlap");
  if (!p->eta_plan) {
    const float c[2] = {e0, e1};
    p->eta_plan = stencil_plan_create(p->nx, p->ny, p->nz, 1, c);
    if (!p->eta_plan) return STENCIL_ERR_CUDA;
  }
  stencil_plan* q = p->eta_plan;
  if (q->c[0] != e0 || q->c[1] != e1) {  // new weights: the launch parameters carry them
    q->c[0] = e0;
    q->c[1] = e1;
    for (int k = 0; k < 5; ++k)
      if (q->kd[k].fn) plan_geometry(q, k);
  }
  return launch(q, 0, eta, nullptr, nullptr, nullptr, eta_eff, static_cast<cudaStream_t>(stream));
}

int stencil_sweeps(stencil_plan* p, float* a, float* b, int nsweeps, int use_graph, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (nsweeps < 0) return fail(STENCIL_ERR_ARG, "nsweeps < 0");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, a, "a")) || (rc = check_field(p, b, "b"))) return rc;
  if (overlap(a, b, (size_t)npoints(p) * 4)) return fail(STENCIL_ERR_ALIAS, "a and b overlap");
  const uint64_t key[8] = {1, (uint64_t)(uintptr_t)a, (uint64_t)(uintptr_t)b, (uint64_t)nsweeps,
                           (uint64_t)p->debug_mode, (uint64_t)p->sweep_path, 0, 0};
  return run_loop(p, key, use_graph != 0, static_cast<cudaStream_t>(stream),
                  [&](cudaStream_t s) { return ping_pong(p, a, b, nsweeps, s); });
}

int wave_steps(stencil_plan* p, float* u_prev, float* u, float* u_tmp, const float* v2dt2,
               const float* eta, int nsteps, int64_t pml_width, int use_graph, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (nsteps < 0) return fail(STENCIL_ERR_ARG, "nsteps < 0");
  int rc = check_device(p);
  if (rc) return rc;
  if ((rc = check_field(p, u_prev, "u_prev")) || (rc = check_field(p, u, "u")) ||
      (rc = check_field(p, u_tmp, "u_tmp")) || (rc = check_field(p, v2dt2, "v2dt2")) ||
      (rc = check_field(p, eta, "eta")))
    return rc;
  const size_t bytes = (size_t)npoints(p) * 4;
  const float* bufs[3] = {u_prev, u, u_tmp};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (overlap(bufs[i], bufs[j], bytes)) return fail(STENCIL_ERR_ALIAS, "time levels overlap");
    if (overlap(bufs[i], v2dt2, bytes) || overlap(bufs[i], eta, bytes))
      return fail(STENCIL_ERR_ALIAS, "a time level overlaps v2dt2 or eta");
  }
  const int64_t pml = pml_width >= 0 ? std::min<int64_t>(pml_width, 1 << 30) : -1;
  const uint64_t key[8] = {2, (uint64_t)(uintptr_t)u_prev, (uint64_t)(uintptr_t)u,
                           (uint64_t)(uintptr_t)u_tmp, (uint64_t)(uintptr_t)v2dt2,
                           (uint64_t)(uintptr_t)eta, ((uint64_t)nsteps << 32) | (uint32_t)(pml + 1),
                           (uint64_t)p->debug_mode};
  return run_loop(p, key, use_graph != 0, static_cast<cudaStream_t>(stream), [&](cudaStream_t s) {
    float* x = u_prev;
    float* y = u;
    float* z = u_tmp;
    for (int i = 0; i < nsteps; ++i) {
      const int r = pml >= 0 ? wave_step_regions(p, x, y, z, v2dt2, eta, pml, s)
                             : launch(p, 1, y, x, v2dt2, eta, z, s);
      if (r) return r;
      float* t = x;  // rotate: (prev, cur, next) <- (cur, next, prev)
      x = y;
      y = z;
      z = t;
    }
    return (int)STENCIL_OK;
  });
}

int stencil_plan_status(stencil_plan* p, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  int rc = check_device(p);
  if (rc) return rc;
  if (p->eta_plan && (rc = stencil_plan_status(p->eta_plan, stream))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned h[4] = {0, 0, 0, 0};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h, p->d_status, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status");
  if (h[0] == 0) return STENCIL_OK;
  e = cudaMemsetAsync(p->d_status, 0, sizeof h, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  if (h[0] & kStatusBadSmem) return fail(STENCIL_ERR_CUDA, "shared memory base misaligned");
  return fail(STENCIL_ERR_TIMEOUT,
              "device wait for staged data ran out (flags 0x%x, block %u, load %u)%s", h[0], h[1],
              h[2], (h[0] & kStatusDrainTimeout) ? "; copies still pending at exit" : "");
}

int stencil_apply_host(stencil_plan* p, const float* in_host, float* out_host, int nsweeps,
                       void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (!in_host || !out_host) return fail(STENCIL_ERR_ARG, "NULL host buffer");
  if (nsweeps < 0) return fail(STENCIL_ERR_ARG, "nsweeps < 0");
  int rc = check_device(p);
  if (rc) return rc;
  const size_t n = (size_t)npoints(p);
  if ((rc = ensure_work(p, 2 * n))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->work;
  float* b = p->work + n;
  if (nsweeps == 1 && !interior_empty(p)) return apply_host_pipelined(p, in_host, out_host, a, b, s);
  cudaError_t e = cudaMemcpyAsync(a, in_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && nsweeps > 0) e = cudaMemcpyAsync(b, a, n * 4, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "copy in");
  if ((rc = ping_pong(p, a, b, nsweeps, s))) return rc;
  if (nsweeps % 2) std::swap(a, b);
  e = cudaMemcpyAsync(out_host, a, n * 4, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "copy out");
  return stencil_plan_status(p, stream);
}

int wave_run_host(stencil_plan* p, float* u_prev_host, float* u_host, const float* v2dt2_host,
                  const float* eta_host, int nsteps, void* stream) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (!u_prev_host || !u_host || !v2dt2_host || !eta_host)
    return fail(STENCIL_ERR_ARG, "NULL host buffer");
  if (nsteps < 0) return fail(STENCIL_ERR_ARG, "nsteps < 0");
  int rc = check_device(p);
  if (rc) return rc;
  const size_t n = (size_t)npoints(p);
  if ((rc = ensure_work(p, 4 * n))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* a = p->work;  // u_prev, then overwritten by u_next (two-buffer stepping)
  float* b = p->work + n;
  float* v = p->work + 2 * n;
  float* et = p->work + 3 * n;
  cudaError_t e = cudaMemcpyAsync(a, u_prev_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(b, u_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v, v2dt2_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(et, eta_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "copy in");
  for (int i = 0; i < nsteps; ++i) {
    if ((rc = launch(p, 1, b, a, v, et, a, s))) return rc;
    std::swap(a, b);
  }
  e = cudaMemcpyAsync(u_prev_host, a, n * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(u_host, b, n * 4, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "copy out");
  return stencil_plan_status(p, stream);
}

int stencil_plan_launch_info(const stencil_plan* p, int kind, int64_t* info, int n) {
  if (!p || !info || n < 0 || kind < 0 || kind > 4) return fail(STENCIL_ERR_ARG, "bad arguments");
  if (!p->kd[kind].fn) return fail(STENCIL_ERR_ARG, "kind %d is not built for radius %d", kind, p->radius);
  const KernelDesc& kd = p->kd[kind];
  const StarParams& sp = p->params[kind];
  int64_t v[11] = {p->grid[kind], kd.threads, kd.smem, p->occupancy[kind], sp.box[0].ntiles,
                   sp.box[0].nchunks, kTX,    kd.tile_y, kd.stages,       p->num_sms, STENCIL_PATH_STAGED};
  if (kind == 0 && p->direct) {  // one thread per 4 x points of an interior row; no tiles or chunks
    int64_t blocks = 0;
    direct_params(p, nullptr, nullptr, 0, (int)(p->nz - 2 * p->radius), blocks);
    const int64_t d[11] = {blocks, kDirectThreads, 0, p->direct_occupancy, 0, 0, 4, 1, 0, p->num_sms,
                           STENCIL_PATH_DIRECT};
    std::copy(d, d + 11, v);
  }
  const int m = std::min(n, 11);
  for (int i = 0; i < m; ++i) info[i] = v[i];
  return m;
}

int stencil_plan_host_phases(const stencil_plan* p, float* ms, int n) {
  if (!p || !ms || n < 0) return fail(STENCIL_ERR_ARG, "bad arguments");
  if (!p->pipe_ready || p->pipe_slabs < 1) return fail(STENCIL_ERR_ARG, "no pipelined host sweep has run");
  const int K = p->pipe_slabs;
  cudaEvent_t start = p->ev[2 * 32], done = p->ev[2 * 32 + 1];
  float v[5] = {0, 0, 0, 0, (float)K};
  cudaError_t e = cudaEventElapsedTime(&v[0], start, done);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&v[1], start, p->ev[0]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&v[2], start, p->ev[K - 1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&v[3], start, p->ev[32 + K - 1]);
  if (e != cudaSuccess) return cuda_fail(e, "host phase events");
  const int m = std::min(n, 5);
  for (int i = 0; i < m; ++i) ms[i] = v[i];
  return m;
}

int stencil_schedule_query(int64_t nx, int64_t ny, int64_t nz, int radius, int kind, int num_sms,
                           int ctas_per_sm, int64_t* info, int n) {
  if (radius < 1 || radius > STENCIL_MAX_RADIUS || kind < 0 || kind > 4 || num_sms < 1 ||
      ctas_per_sm < 1 || !info || n < 0)
    return fail(STENCIL_ERR_ARG, "bad arguments");
  if (nx < 1 || ny < 1 || nz < 1 || nx > (1 << 30) || ny > (1 << 30) || nz > (1 << 30) ||
      nx * ny > ((int64_t)1 << 40) || nx * ny * nz > ((int64_t)1 << 40))
    return fail(STENCIL_ERR_ARG, "grid %lld x %lld x %lld out of range", (long long)nx,
                (long long)ny, (long long)nz);
  const KernelDesc kd = kind == 0   ? apply_kernel_desc(radius, nx, ny)
                        : kind == 3 ? semi_kernel_desc(radius)
                        : kind == 4 ? apply2_kernel_desc(radius)
                                    : wave_kernel_desc(radius, kind == 2);
  if (!kd.fn) return fail(STENCIL_ERR_ARG, "kind %d is not built for radius %d", kind, radius);
  const int64_t m = 2 * (int64_t)radius + 1;
  Schedule sc{};
  if (nx >= m && ny >= m && nz >= m)
    sc = schedule(nx, ny, radius, kd.tile_y, kind, num_sms, ctas_per_sm, (int)(nz - 2 * radius), kd.tstore);
  const int64_t v[7] = {sc.grid, sc.ntiles, sc.nchunks, sc.nitems, kTX, kd.tile_y, kd.tstore ? radius : 0};
  const int k = std::min(n, 7);
  for (int i = 0; i < k; ++i) info[i] = v[i];
  return k;
}

int stencil_plan_set_sweep_path(stencil_plan* p, int path) {
  if (!p) return fail(STENCIL_ERR_ARG, "plan is NULL");
  if (path < STENCIL_PATH_AUTO || path > STENCIL_PATH_DIRECT)
    return fail(STENCIL_ERR_ARG, "sweep path %d is not one of 0 (auto), 1 (staged), 2 (direct)", path);
  p->sweep_path = path;
  p->direct = resolve_direct(p);
  return STENCIL_OK;
}

int stencil_debug_inject(stencil_plan* p, int mode) {
  if (!p || mode < 0 || mode > 1) return fail(STENCIL_ERR_ARG, "bad arguments");
  p->debug_mode = mode;
  return STENCIL_OK;
}

}  // extern "C"

// ---- allocation-free sweep ---------------------------------------------------------
//
// Some callers cannot allocate device memory at the time they need a sweep: code that
// runs inside another framework's memory pool which owns all free device memory, or a
// process whose device-memory footprint is fixed at start-up.  For them,
// stencil_apply_noalloc runs the same sweep kernel as stencil_apply, with the kernel's
// status block placed in the file-scope device array below instead of plan-owned
// memory, and builds its plan on the stack.
//
// In host code `g_noalloc_scratch` names a host-side stand-in, not the device copy:
// passing it to a kernel would fault (or, where the GPU can reach host memory, silently
// use the wrong memory).  Every call asks cudaGetSymbolAddress for the array's address
// in the current device's context (a lookup, no allocation); nothing is cached, so a
// context that was reset and re-created since the previous call gets its own address.
namespace {

constexpr int kNoAllocScratchWords = 64;  // 256 bytes; the sweep uses the first 4 words
__device__ __align__(256) unsigned g_noalloc_scratch[kNoAllocScratchWords];

int noalloc_scratch(unsigned** out) {
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
  *out = static_cast<unsigned*>(ptr);
  return STENCIL_OK;
}

}  // namespace

extern "C" int stencil_apply_noalloc(int64_t nx, int64_t ny, int64_t nz, int radius,
                                     const float* coeffs, const float* in, float* out,
                                     void* stream) {
  g_err[0] = 0;
  if (radius < 1 || radius > STENCIL_MAX_RADIUS)
    return fail(STENCIL_ERR_ARG, "radius %d outside [1, %d]", radius, STENCIL_MAX_RADIUS);
  if (!coeffs) return fail(STENCIL_ERR_ARG, "coeffs is NULL");
  if (nx < 1 || ny < 1 || nz < 1 || nx > (1 << 30) || ny > (1 << 30) || nz > (1 << 30) ||
      nx * ny > ((int64_t)1 << 40) || nx * ny * nz > ((int64_t)1 << 40))
    return fail(STENCIL_ERR_ARG,
                "grid %lld x %lld x %lld beyond the maximum (each dimension <= 2^30, at most "
                "2^40 points)",
                (long long)nx, (long long)ny, (long long)nz);
  if (nx % 4) return fail(STENCIL_ERR_ALIGNMENT, "nx = %lld is not a multiple of 4", (long long)nx);

  stencil_plan pl{};  // on the stack: no heap or device allocation
  pl.nx = nx;
  pl.ny = ny;
  pl.nz = nz;
  pl.radius = radius;
  for (int r = 0; r <= STENCIL_MAX_RADIUS; ++r) pl.c[r] = r <= radius ? coeffs[r] : 0.0f;
  cudaError_t e = cudaGetDevice(&pl.device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&pl.num_sms, cudaDevAttrMultiProcessorCount, pl.device);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  int rc = noalloc_scratch(&pl.d_status);
  if (rc) return rc;
  pl.kd[0] = apply_kernel_desc(radius, nx, ny);
  e = cudaFuncSetAttribute(pl.kd[0].fn, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.kd[0].smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pl.occupancy[0], pl.kd[0].fn,
                                                      pl.kd[0].threads, pl.kd[0].smem);
  if (e != cudaSuccess) return cuda_fail(e, "kernel attributes");
  if (pl.occupancy[0] < 1) return fail(STENCIL_ERR_CUDA, "kernel cannot be resident (occupancy 0)");
  plan_geometry(&pl, 0);
  pl.sweep_path = STENCIL_PATH_AUTO;
  pl.direct = resolve_direct(&pl);

  if ((rc = check_field(&pl, in, "in")) || (rc = check_field(&pl, out, "out"))) return rc;
  if (overlap(in, out, (size_t)npoints(&pl) * 4)) return fail(STENCIL_ERR_ALIAS, "in and out overlap");

  // The scratch keeps the previous call's contents: clear the status words first.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(pl.d_status, 0, 4 * sizeof(unsigned), s);
  if (e != cudaSuccess) return cuda_fail(e, "clear scratch");
  if ((rc = launch(&pl, 0, in, nullptr, nullptr, nullptr, out, s))) return rc;
  unsigned h[4] = {0, 0, 0, 0};
  e = cudaMemcpyAsync(h, pl.d_status, sizeof h, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "sweep");
  if (h[0] & kStatusBadSmem) return fail(STENCIL_ERR_CUDA, "shared memory base misaligned");
  if (h[0])
    return fail(STENCIL_ERR_TIMEOUT, "device wait for staged data ran out (flags 0x%x, block %u, load %u)",
                h[0], h[1], h[2]);
  return STENCIL_OK;
}

// ---- z-slab decomposition ----------------------------------------------------------
//
// The grid is cut along z into slabs; slab k owns the global planes [o_k, o_k+1) and
// stores them with up to R ghost planes on each side, [s_k, e_k) = [max(0, o_k - R),
// min(nz, o_k+1 + R)), as an nx x ny x (e_k - s_k) array of its own.  Its local interior
// is then exactly its owned interior planes, so a sweep of the whole grid is one sweep
// per slab once every ghost plane holds its owner's current values.  The exchange is one
// copy of R planes each way per cut; the output planes that read no ghost plane run
// while the copies are in flight, the 2R planes next to each cut after them.
struct stencil_slabs {
  int64_t nx, ny, nz;
  int radius;
  int nslabs;
  int device;
  std::vector<int64_t> own;           // o_0 .. o_P
  std::vector<stencil_plan*> plans;   // one per slab, for its stored planes
  cudaStream_t copy;                  // the exchange's stream
  cudaEvent_t fork, join;
};

namespace {

int64_t slab_begin(const stencil_slabs* S, int k) { return std::max<int64_t>(0, S->own[k] - S->radius); }
int64_t slab_end(const stencil_slabs* S, int k) { return std::min<int64_t>(S->nz, S->own[k + 1] + S->radius); }

int check_slab_fields(stencil_slabs* S, float* const* f, const char* name) {
  if (!f) return fail(STENCIL_ERR_ARG, "%s is NULL", name);
  for (int k = 0; k < S->nslabs; ++k) {
    char what[64];
    snprintf(what, sizeof what, "%s[%d]", name, k);
    const int rc = check_field(S->plans[k], f[k], what);
    if (rc) return rc;
  }
  return STENCIL_OK;
}

size_t slab_bytes(const stencil_slabs* S, int k) {
  return (size_t)(S->nx * S->ny * (slab_end(S, k) - slab_begin(S, k))) * 4;
}

// No two of the listed slab arrays may overlap (one field's slabs, or two fields).
int check_slab_overlaps(const stencil_slabs* S, float* const* const* fields, int nfields) {
  for (int f = 0; f < nfields; ++f)
    for (int g = f; g < nfields; ++g)
      for (int j = 0; j < S->nslabs; ++j)
        for (int k = (f == g ? j + 1 : 0); k < S->nslabs; ++k) {
          const float* a = fields[f][j];
          const float* b = fields[g][k];
          const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
          if (x < y + slab_bytes(S, k) && y < x + slab_bytes(S, j))
            return fail(STENCIL_ERR_ALIAS, "slab arrays overlap (field %d slab %d, field %d slab %d)", f,
                        j, g, k);
        }
  return STENCIL_OK;
}

// Ghost copies of every cut on stream s: slab c-1's top ghosts from slab c's first owned
// planes, slab c's bottom ghosts from slab c-1's last owned planes.
int slab_exchange(stencil_slabs* S, float* const* f, cudaStream_t s) {
  const int R = S->radius;
  const size_t plane = (size_t)S->nx * S->ny;
  for (int c = 1; c < S->nslabs; ++c) {
    const int64_t cut = S->own[c];
    const int64_t lo = slab_begin(S, c - 1), hi = slab_begin(S, c);
    cudaError_t e = cudaMemcpyAsync(f[c - 1] + (size_t)(cut - lo) * plane, f[c] + (size_t)(cut - hi) * plane,
                                    (size_t)R * plane * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(f[c] + (size_t)(cut - R - hi) * plane, f[c - 1] + (size_t)(cut - R - lo) * plane,
                          (size_t)R * plane * 4, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "ghost exchange");
  }
  return STENCIL_OK;
}

// One sweep (kind 0) or wave step (kind 1) of every slab: the exchange of `x` (the field
// the stencil reads) on the exchange stream, overlapped with the output planes that read
// no ghost plane; then the planes next to the cuts.
int slab_run(stencil_slabs* S, int kind, float* const* x, float* const* uprev, float* const* v2dt2,
             float* const* eta, float* const* out, cudaStream_t s) {
  const int R = S->radius;
  const int P = S->nslabs;
  // Local output-plane ranges per slab: [a, b) first, then the dependent ranges.
  std::vector<int64_t> in_lo(P), in_hi(P);
  for (int k = 0; k < P; ++k) {
    const int64_t nzk = slab_end(S, k) - slab_begin(S, k);
    in_lo[k] = k > 0 ? 2 * R : R;
    in_hi[k] = k < P - 1 ? nzk - 2 * R : nzk - R;
    if (in_hi[k] - in_lo[k] < R) in_lo[k] = in_hi[k] = R;  // too thin to split: all after the copies
  }
  auto run = [&](int k, int64_t lo, int64_t hi, cudaStream_t st) {
    if (hi <= lo) return (int)STENCIL_OK;
    stencil_plan* p = S->plans[k];
    return launch(p, kind, x[k], uprev ? uprev[k] : nullptr, v2dt2 ? v2dt2[k] : nullptr,
                  eta ? eta[k] : nullptr, out[k], st, (int)(lo - R), (int)(hi - lo));
  };
  if (P > 1) {
    cudaError_t e = cudaEventRecord(S->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(S->copy, S->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "exchange fork");
  }
  for (int k = 0; k < P; ++k) {
    const int rc = run(k, in_lo[k], in_hi[k], s);
    if (rc) return rc;
  }
  // The planes next to the cuts follow the copies on the exchange stream, so they run
  // alongside the interior launches instead of after them.
  cudaStream_t bs = P > 1 ? S->copy : s;
  if (P > 1) {
    const int rc = slab_exchange(S, x, bs);
    if (rc) return rc;
  }
  for (int k = 0; k < P; ++k) {
    const int64_t nzk = slab_end(S, k) - slab_begin(S, k);
    int rc;
    if (in_hi[k] <= in_lo[k]) {
      rc = run(k, R, nzk - R, bs);
    } else {
      rc = run(k, R, in_lo[k], bs);
      if (!rc) rc = run(k, in_hi[k], nzk - R, bs);
    }
    if (rc) return rc;
  }
  if (P > 1) {
    cudaError_t e = cudaEventRecord(S->join, bs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, S->join, 0);
    if (e != cudaSuccess) return cuda_fail(e, "exchange join");
  }
  return STENCIL_OK;
}

}  // namespace

extern "C" {

stencil_slabs* stencil_slabs_create(int64_t nx, int64_t ny, int64_t nz, int radius, const float* coeffs,
                                    int nslabs) {
  g_err[0] = 0;
  if (nslabs < 1) {
    fail(STENCIL_ERR_ARG, "nslabs %d < 1", nslabs);
    return nullptr;
  }
  if (radius >= 1 && nz / nslabs < radius) {
    fail(STENCIL_ERR_ARG, "%d slabs of %lld planes: every slab must own at least radius = %d planes",
         nslabs, (long long)nz, radius);
    return nullptr;
  }
  stencil_slabs* S = new stencil_slabs();
  S->nx = nx;
  S->ny = ny;
  S->nz = nz;
  S->radius = radius;
  S->nslabs = nslabs;
  for (int k = 0; k <= nslabs; ++k) S->own.push_back(nz * k / nslabs);
  for (int k = 0; k < nslabs; ++k) {
    stencil_plan* p = stencil_plan_create(nx, ny, slab_end(S, k) - slab_begin(S, k), radius, coeffs);
    if (!p) {
      stencil_slabs_destroy(S);
      return nullptr;
    }
    S->plans.push_back(p);
  }
  S->device = S->plans[0]->device;
  cudaError_t e = cudaStreamCreateWithFlags(&S->copy, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&S->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&S->join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cuda_fail(e, "slab streams");
    stencil_slabs_destroy(S);
    return nullptr;
  }
  return S;
}

void stencil_slabs_destroy(stencil_slabs* S) {
  if (!S) return;
  for (stencil_plan* p : S->plans) stencil_plan_destroy(p);
  if (S->copy) cudaStreamDestroy(S->copy);
  if (S->fork) cudaEventDestroy(S->fork);
  if (S->join) cudaEventDestroy(S->join);
  delete S;
}

int stencil_slabs_extent(const stencil_slabs* S, int k, int64_t* info, int n) {
  if (!S || !info || n < 0 || k < 0 || k >= S->nslabs) return fail(STENCIL_ERR_ARG, "bad arguments");
  const int64_t v[4] = {slab_begin(S, k), slab_end(S, k), S->own[k], S->own[k + 1]};
  const int m = std::min(n, 4);
  for (int i = 0; i < m; ++i) info[i] = v[i];
  return m;
}

int stencil_slabs_exchange(stencil_slabs* S, float* const* fields, void* stream) {
  if (!S) return fail(STENCIL_ERR_ARG, "slabs is NULL");
  int rc = check_device(S->plans[0]);
  if (rc || (rc = check_slab_fields(S, fields, "fields"))) return rc;
  float* const* all[1] = {fields};
  if ((rc = check_slab_overlaps(S, all, 1))) return rc;
  return slab_exchange(S, fields, static_cast<cudaStream_t>(stream));
}

int stencil_slabs_apply(stencil_slabs* S, float* const* in, float* const* out, void* stream) {
  if (!S) return fail(STENCIL_ERR_ARG, "slabs is NULL");
  int rc = check_device(S->plans[0]);
  if (rc || (rc = check_slab_fields(S, in, "in")) || (rc = check_slab_fields(S, out, "out"))) return rc;
  float* const* all[2] = {in, out};
  if ((rc = check_slab_overlaps(S, all, 2))) return rc;
  return slab_run(S, 0, in, nullptr, nullptr, nullptr, out, static_cast<cudaStream_t>(stream));
}

int stencil_slabs_wave_step(stencil_slabs* S, float* const* u_prev, float* const* u, float* const* u_next,
                            float* const* v2dt2, float* const* eta, void* stream) {
  if (!S) return fail(STENCIL_ERR_ARG, "slabs is NULL");
  int rc = check_device(S->plans[0]);
  if (rc || (rc = check_slab_fields(S, u_prev, "u_prev")) || (rc = check_slab_fields(S, u, "u")) ||
      (rc = check_slab_fields(S, u_next, "u_next")) || (rc = check_slab_fields(S, v2dt2, "v2dt2")) ||
      (rc = check_slab_fields(S, eta, "eta")))
    return rc;
  // u_next == u_prev (every slab) is allowed, as for wave_step.
  const bool two_buffers = u_next[0] == u_prev[0];
  for (int k = 0; k < S->nslabs; ++k)
    if ((u_next[k] == u_prev[k]) != two_buffers)
      return fail(STENCIL_ERR_ALIAS, "u_next equals u_prev for some slabs only");
  if (two_buffers) {
    float* const* all[4] = {u, u_next, v2dt2, eta};
    if ((rc = check_slab_overlaps(S, all, 4))) return rc;
  } else {
    float* const* all[5] = {u_prev, u, u_next, v2dt2, eta};
    if ((rc = check_slab_overlaps(S, all, 5))) return rc;
  }
  return slab_run(S, 1, u, u_prev, v2dt2, eta, u_next, static_cast<cudaStream_t>(stream));
}

int stencil_slabs_status(stencil_slabs* S, void* stream) {
  if (!S) return fail(STENCIL_ERR_ARG, "slabs is NULL");
  for (stencil_plan* p : S->plans) {
    const int rc = stencil_plan_status(p, stream);
    if (rc) return rc;
  }
  return STENCIL_OK;
}

}  // extern "C"
