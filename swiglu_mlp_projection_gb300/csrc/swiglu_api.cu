// C ABI of the SwiGLU up-projection library: validation, dispatch, workspace.
//
// Everything a call does on the GPU runs in the kernels of this directory; this
// file only checks arguments, chooses a path and enqueues the launches on the
// caller's stream.  See include/swiglu.h for the contract of each entry point.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>   // environ

#include "swiglu.h"
#include "common.cuh"
#include "internal.h"

namespace swg {

// Error word written by bounded device-side waits that give up.
__device__ unsigned g_device_status = 0;

namespace {

thread_local char t_err[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof t_err, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SWIGLU_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int max_pairs = 0;            // 2-CTA clusters of the tile kernel that fit at once
  int sk_caps[4] = {0, 0, 0, 0};   // clusters of 2, 4, 8 skinny CTAs that fit at once
  int simt_caps[kSimtCapSlots] = {};   // clusters of S SIMT-cluster CTAs that fit at once
  int cc_major = 0, cc_minor = 0;
  cudaMemPool_t pool = nullptr;
  unsigned* status = nullptr;   // device address of g_device_status
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Fills `out` for the current device (cached).  Returns a swiglu_status.
int current_device(int* dev_out, DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    if ((e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    if ((e = cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(cc major)");
    if ((e = cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(cc minor)");
    if (di.cc_major == 10 && di.cc_minor == 3) {
      void* sp = nullptr;
      if ((e = cudaGetSymbolAddress(&sp, g_device_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(status word)");
      di.status = (unsigned*)sp;
      if ((e = tile_max_pairs(&di.max_pairs)) != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters(tile kernel)");
      if ((e = skinny_cluster_caps(di.sk_caps)) != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters(skinny kernel)");
      if ((e = simt_cluster_caps(di.simt_caps)) != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveClusters(SIMT cluster kernel)");
    }
    di.ready = true;
  }
  *dev_out = dev;
  *out = di;
  if (di.cc_major != 10 || di.cc_minor != 3)
    return fail(SWIGLU_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, di.cc_major, di.cc_minor);
  return SWIGLU_OK;
}

// The library's stream-ordered workspace pool for `dev` (created on first use;
// it keeps freed blocks for reuse instead of returning them to the driver).
int device_pool(int dev, cudaMemPool_t* pool) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.pool) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&di.pool, &props);
    if (e != cudaSuccess) { di.pool = nullptr; return cuda_fail(e, "cudaMemPoolCreate"); }
    uint64_t keep = ~0ull;
    e = cudaMemPoolSetAttribute(di.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolSetAttribute");
  }
  *pool = di.pool;
  return SWIGLU_OK;
}

// Library-owned workspace, kept per stream.  Layout: kStreamCounterBytes of
// arrival counters for the skinny kernel, then the partial sums of either
// split-K path.  Calls on one stream run in stream order, so they can share
// the buffer; the skinny kernel leaves every counter it used at zero, so the
// next call needs no clearing.  Streams are told apart by cudaStreamGetId,
// which is never reused within a process.  Counters of a call that gave up
// may be left non-zero: swiglu_check_device_status marks the device's
// buffers dirty and the next call clears their counters.  The buffer grows
// (stream-ordered free of the old one) when a call needs more.
struct StreamWorkspace {
  int dev;
  unsigned long long stream_id;
  char* base;
  size_t part_capacity;
  bool dirty;
};
constexpr size_t kMaxStreamSlots = 256;
constexpr size_t kMaxCachedPartBytes = (size_t)256 << 20;
std::vector<StreamWorkspace> g_stream_ws;   // guarded by g_mu

int device_pool(int dev, cudaMemPool_t* pool);

// On success, either *part (and *counters, already zero) point into the
// stream's buffer, or both are null and the call must bring its own
// workspace: the per-thread default stream (its handle is shared by threads
// that are not ordered with each other), a stream without an id, too many
// streams, or a very large request.
int stream_workspace(int dev, cudaStream_t st, size_t part_bytes, float** part,
                     unsigned** counters) {
  *part = nullptr;
  *counters = nullptr;
  if (st == cudaStreamPerThread || part_bytes > kMaxCachedPartBytes) return SWIGLU_OK;
  // A call being captured into a CUDA graph does not use this stream's
  // buffer: a replay may run on another stream, unordered with later calls
  // that would share it.  It takes its capture's slice (graph_workspace).
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_OK;
  }
  if (cs != cudaStreamCaptureStatusNone) return SWIGLU_OK;
  unsigned long long id = 0;
  if (cudaStreamGetId(st, &id) != cudaSuccess) {
    cudaGetLastError();
    return SWIGLU_OK;
  }
  cudaMemPool_t pool;
  int v = device_pool(dev, &pool);
  if (v != SWIGLU_OK) return v;
  std::lock_guard<std::mutex> lk(g_mu);
  StreamWorkspace* sw = nullptr;
  for (auto& e : g_stream_ws)
    if (e.dev == dev && e.stream_id == id) sw = &e;
  if (!sw) {
    if (g_stream_ws.size() >= kMaxStreamSlots) return SWIGLU_OK;
    g_stream_ws.push_back({dev, id, nullptr, 0, true});
    sw = &g_stream_ws.back();
  }
  if (!sw->base || sw->part_capacity < part_bytes) {
    const size_t cap = (part_bytes + ((size_t)1 << 20) - 1) & ~(((size_t)1 << 20) - 1);
    void* p = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&p, kStreamCounterBytes + cap, pool, st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return SWIGLU_OK;   // the call falls back to a per-call workspace
    }
    if (sw->base) cudaFreeAsync(sw->base, st);
    sw->base = (char*)p;
    sw->part_capacity = cap;
    sw->dirty = true;
  }
  if (sw->dirty) {
    cudaError_t e = cudaMemsetAsync(sw->base, 0, kStreamCounterBytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(counters)");
    sw->dirty = false;
  }
  *counters = (unsigned*)sw->base;
  *part = (float*)(sw->base + kStreamCounterBytes);
  return SWIGLU_OK;
}

void mark_workspaces_dirty(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_stream_ws)
    if (e.dev == dev) e.dirty = true;
}

// Drops the cached buffer of stream `st` on `dev`: a stream-ordered free on
// `st` itself, after the work already enqueued there.
int release_stream_workspace(int dev, cudaStream_t st) {
  if (st == cudaStreamPerThread) return SWIGLU_OK;   // never cached
  unsigned long long id = 0;
  cudaError_t e = cudaStreamGetId(st, &id);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetId");
  std::lock_guard<std::mutex> lk(g_mu);
  for (size_t i = 0; i < g_stream_ws.size(); ++i) {
    StreamWorkspace& w = g_stream_ws[i];
    if (w.dev != dev || w.stream_id != id) continue;
    if (w.base && (e = cudaFreeAsync(w.base, st)) != cudaSuccess)
      return cuda_fail(e, "cudaFreeAsync(stream workspace)");
    g_stream_ws.erase(g_stream_ws.begin() + (ptrdiff_t)i);
    break;
  }
  return SWIGLU_OK;
}

// Drops every cached buffer of `dev` once the device is idle, and returns the
// pool's unused memory to the driver.  Buffers of streams the caller has
// destroyed are freed too: no stream handle is needed.
int release_device_workspaces(int dev) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (size_t i = 0; i < g_stream_ws.size();) {
      StreamWorkspace& w = g_stream_ws[i];
      if (w.dev != dev) { ++i; continue; }
      if (w.base && (e = cudaFreeAsync(w.base, cudaStreamLegacy)) != cudaSuccess)
        return cuda_fail(e, "cudaFreeAsync(stream workspace)");
      g_stream_ws.erase(g_stream_ws.begin() + (ptrdiff_t)i);
    }
    pool = g_dev[dev].pool;
  }
  if ((e = cudaStreamSynchronize(cudaStreamLegacy)) != cudaSuccess)
    return cuda_fail(e, "cudaStreamSynchronize");
  if (pool && (e = cudaMemPoolTrimTo(pool, 0)) != cudaSuccess)
    return cuda_fail(e, "cudaMemPoolTrimTo");
  return SWIGLU_OK;
}

size_t cached_workspace_bytes(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  size_t n = 0;
  for (const auto& w : g_stream_ws)
    if (w.dev == dev && w.base) n += kStreamCounterBytes + w.part_capacity;
  return n;
}

// Arrival counters for calls captured into CUDA graphs.  A captured call's
// workspace is a graph allocation whose contents are undefined on every
// replay, so its counters would need a memset node, which costs ~5 us per
// d = 4096 decode call and breaks the programmatic overlap with the previous
// kernel.  Instead each captured call takes its own counters, once, from a
// per-device region zeroed when it was created; the kernels leave them at
// zero, so every replay finds them clean.  Slices are never reused: graphs
// replay independently of each other (a graph exec never overlaps itself).
// The region is created by the first non-captured call that uses counters
// (one synchronisation of that call's stream); captures made before it, or
// after it fills up, fall back to allocating and clearing.
struct GraphCounters {
  char* base = nullptr;
  size_t cap = 0, used = 0;
  bool tried = false;
};
GraphCounters g_gctr[kMaxDevices];   // guarded by g_mu
constexpr size_t kGraphCounterBytes = (size_t)4 << 20;

void ensure_graph_counters(int dev, cudaStream_t st) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_gctr[dev].tried) return;
    g_gctr[dev].tried = true;
  }
  cudaMemPool_t pool;
  if (device_pool(dev, &pool) != SWIGLU_OK) return;
  void* p = nullptr;
  if (cudaMallocFromPoolAsync(&p, kGraphCounterBytes, pool, st) != cudaSuccess ||
      cudaMemsetAsync(p, 0, kGraphCounterBytes, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_gctr[dev].base = (char*)p;
  g_gctr[dev].cap = kGraphCounterBytes;
}

// Workspaces of calls captured into CUDA graphs.  A workspace that the
// capture itself allocates (cudaMallocFromPoolAsync on the capturing stream)
// puts allocation and free nodes between the kernel nodes, and they cut the
// programmatic overlap of consecutive calls: a d = 4096 decode call replays
// in 40.7 us that way, against 37.1 us with its workspace allocated outside
// the graph (37.5 us back to back on a stream).  So a captured call takes a
// workspace that this thread allocates outside the graph (in relaxed capture
// mode) and zeroes once: one slice per capture sequence and capturing stream,
// reused by that capture's later calls on that stream.  Those run one after
// another (each call's kernels wait for the previous kernel in the stream
// before they touch the workspace) and leave its arrival counters at zero.
// Slices live as long as the process, since a graph may be replayed at any
// time, and one graph exec never overlaps itself.  A capture that would take
// the slices past kMaxGraphWorkspaceBytes falls back to allocation nodes.
struct GraphSlice {
  int dev;
  unsigned long long capture_id;
  uintptr_t stream;
  char* base;
  size_t bytes;
};
std::vector<GraphSlice> g_graph_ws;        // guarded by g_mu
size_t g_graph_ws_bytes[kMaxDevices] = {};  // guarded by g_mu
cudaStream_t g_graph_ws_stream[kMaxDevices] = {};   // zeroes new slices; guarded by g_mu
constexpr size_t kMaxGraphWorkspaceBytes = (size_t)8 << 30;

// A zeroed workspace of at least `bytes` for the call being captured on
// `st`, or null (the caller then allocates inside the graph).
char* graph_workspace(int dev, cudaStream_t st, size_t bytes) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  unsigned long long id = 0;
  if (cudaStreamGetCaptureInfo(st, &cs, &id) != cudaSuccess ||
      cs != cudaStreamCaptureStatusActive) {
    cudaGetLastError();
    return nullptr;
  }
  bytes = (bytes + 255) / 256 * 256;
  std::lock_guard<std::mutex> lk(g_mu);
  for (const GraphSlice& g : g_graph_ws)
    if (g.dev == dev && g.capture_id == id && g.stream == (uintptr_t)st && g.bytes >= bytes)
      return g.base;
  if (g_graph_ws_bytes[dev] + bytes > kMaxGraphWorkspaceBytes) return nullptr;
  // Allocate and clear outside the graph: this thread may make those calls
  // while a stream captures only in relaxed mode.
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  void* p = nullptr;
  cudaError_t e = cudaSuccess;
  if (!g_graph_ws_stream[dev])
    e = cudaStreamCreateWithFlags(&g_graph_ws_stream[dev], cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaMalloc(&p, bytes);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, bytes, g_graph_ws_stream[dev]);
  if (e == cudaSuccess) e = cudaStreamSynchronize(g_graph_ws_stream[dev]);
  if (e != cudaSuccess && p) {
    cudaFree(p);
    p = nullptr;
  }
  cudaThreadExchangeStreamCaptureMode(&mode);   // back to the caller's mode
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  g_graph_ws.push_back({dev, id, (uintptr_t)st, (char*)p, bytes});
  g_graph_ws_bytes[dev] += bytes;
  return (char*)p;
}

unsigned* take_graph_counters(int dev, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  GraphCounters& g = g_gctr[dev];
  bytes = (bytes + 255) / 256 * 256;
  if (!g.base || g.used + bytes > g.cap) return nullptr;
  unsigned* r = (unsigned*)(g.base + g.used);
  g.used += bytes;
  return r;
}

int elem_bytes(int dtype) { return dtype == SWIGLU_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

// Largest bf16 M that AUTO sends to the skinny kernel, by operation and by
// the skinny kernel's mode for the weights: cluster mode (at most 32 MB) or
// stream-K.  The decode article serves at most 16 rows with its skinny
// kernel; the tcgen05 skinny kernel pays longer.
constexpr int64_t kSkinnyMaxM = 32;
constexpr int64_t kSkinnyMaxMSmall = 128;
constexpr int64_t kSkinnyMaxMDown = 256;

// Grid-dimension limits of the SIMT path (gridDim.y/z are 16-bit).
constexpr int64_t kMaxGridYZ = kSimtMaxGridYZ;

// Bound of every device-side wait, from SWIGLU_WAIT_TIMEOUT_MS (default 2 s).
uint64_t wait_timeout_ns() {
  static uint64_t ns = [] {
    const char* v = getenv("SWIGLU_WAIT_TIMEOUT_MS");
    long long ms = v ? atoll(v) : 0;
    if (ms <= 0) ms = 2000;
    return (uint64_t)ms * 1000000ull;
  }();
  return ns;
}

// The two operations the library serves.
enum Op { kOpUp = 0, kOpDown = 1 };

// The measured crossovers (both paths forced, calls back to back, residual
// included).  Stream-K mode: up projection 32 at d = 4096 and 8192 (d =
// 4096: 39.4 vs 40.2 us at M = 32, 42.8 vs 40.4 at 48); down projection,
// with its sums in a second kernel, all the 256 rows the kernel serves (d =
// 4096: 32.3 vs 50.3 us at M = 256; d = 8192: 83.3 vs 111.3 at 128, 100.7
// vs 143.9 at 256; FP8 d = 4096: 27.2 vs 45.6 at 256).  Cluster mode, d =
// 896 (graph replay; 64-column groups from 16 rows): up projection 128
// (9.97 vs 10.67 us at M = 128, 11.84 vs 10.39 at 192); down projection
// all M the kernel serves (13.9 vs 27.3 us at M = 256).  FP8 calls measure
// alike otherwise.
int64_t skinny_max_m(int op, int64_t K, int64_t n_out, int num_sms, const int* sk_caps) {
  const bool small = (op == kOpDown ? 1 : 2) * K * n_out * 2 <= kSkinnyClusterMaxWeightBytes;
  (void)num_sms;
  (void)sk_caps;
  if (op == kOpDown) return kSkinnyMaxMDown;
  return small ? kSkinnyMaxMSmall : kSkinnyMaxM;
}

}  // namespace

Tuning read_tuning() {
  Tuning t;
  for (char** e = environ; e && *e; ++e) {
    const char* s = *e;
    if (strncmp(s, "SWIGLU_", 7) != 0) continue;
    const char* eq = strchr(s, '=');
    if (!eq) continue;
    const char* name = s + 7;
    const size_t n = (size_t)(eq - name);
    const int v = atoi(eq + 1);
    struct Knob { const char* key; int* dst; };
    const Knob knobs[] = {{"SK_NB", &t.sk_nb},
                          {"SK_PROMO", &t.sk_promo},
                          {"SK_HINT", &t.sk_hint},
                          {"SK_PREFETCH_UNITS", &t.sk_prefetch_units},
                          {"SK_CLUSTER", &t.sk_cluster},
                          {"TILE_PAIR", &t.tile_pair},
                          {"TILE_SK", &t.tile_sk},
                          {"TILE_SK_SPLIT", &t.tile_sk_split},
                          {"TILE_SEQ", &t.tile_seq},
                          {"TILE_BAND", &t.tile_band},
                          {"SIMT_FUSED", &t.simt_fused},
                          {"SK_BULK", &t.sk_bulk},
                          {"SK_SPLIT", &t.sk_split},
                          {"SK_KB", &t.sk_kb},
                          {"SIMT_CLUSTER", &t.simt_cluster},
                          {"INJECT_OOM", &t.inject_oom}};
    for (const Knob& k : knobs)
      if (strlen(k.key) == n && strncmp(k.key, name, n) == 0) *k.dst = v;
  }
  return t;
}

namespace {

// Up projection, AUTO: f32 -> SIMT; bf16 M <= skinny_max_m -> SKINNY; larger
// bf16 M -> TC.  d == 0 (empty sums) always goes to the SIMT path, whose
// reduction kernel then writes h = silu(0) * 0 = 0.
// Down projection: bf16 only, on the tensor-core paths (M <= skinny_max_m
// -> SKINNY).
int resolve_path(int op, int64_t M, int64_t K, int64_t n_out, int dtype, int path, int* out,
                 int num_sms, const int* sk_caps) {
  if (path < SWIGLU_PATH_AUTO || path > SWIGLU_PATH_TC)
    return fail(SWIGLU_ERR_INVALID_ARG, "unknown path %d", path);
  if (op == kOpDown) {
    if (dtype != SWIGLU_BF16)
      return fail(SWIGLU_ERR_UNSUPPORTED, "the down projection serves bf16 only");
    if (path == SWIGLU_PATH_SIMT)
      return fail(SWIGLU_ERR_UNSUPPORTED, "the down projection has no SIMT path");
  }
  if (path == SWIGLU_PATH_AUTO) {
    if (op == kOpUp && (dtype == SWIGLU_F32 || K == 0)) *out = SWIGLU_PATH_SIMT;
    else
      *out = M <= skinny_max_m(op, K, n_out, num_sms, sk_caps) ? SWIGLU_PATH_SKINNY
                                                                : SWIGLU_PATH_TC;
    return SWIGLU_OK;
  }
  if (path != SWIGLU_PATH_SIMT && dtype != SWIGLU_BF16)
    return fail(SWIGLU_ERR_UNSUPPORTED, "the tensor-core paths serve bf16 only");
  if (path == SWIGLU_PATH_SKINNY && M > kSkinnyMaxN)
    return fail(SWIGLU_ERR_UNSUPPORTED, "the skinny path serves M <= %d", kSkinnyMaxN);
  *out = (op == kOpUp && K == 0) ? SWIGLU_PATH_SIMT : path;
  return SWIGLU_OK;
}

int check_sizes(int64_t M, int64_t d, int64_t d_ff, int dtype) {
  if (dtype != SWIGLU_F32 && dtype != SWIGLU_BF16)
    return fail(SWIGLU_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (M < 0 || d < 0 || d_ff < 0)
    return fail(SWIGLU_ERR_INVALID_ARG, "negative size (M=%lld d=%lld d_ff=%lld)",
                (long long)M, (long long)d, (long long)d_ff);
  if (M > INT32_MAX || d > INT32_MAX || d_ff > INT32_MAX)
    return fail(SWIGLU_ERR_UNSUPPORTED, "a size exceeds 2^31-1");
  const int64_t per16 = (int64_t)(16 / elem_bytes(dtype));
  if (d % per16 != 0 || d_ff % per16 != 0)
    return fail(SWIGLU_ERR_ALIGNMENT, "d and d_ff must be multiples of %lld for this dtype",
                (long long)per16);
  return SWIGLU_OK;
}

int validate(const void* x, const void* wg, const void* wu, const void* h,
             int64_t M, int64_t d, int64_t d_ff, int dtype) {
  int v = check_sizes(M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  const size_t e = (size_t)elem_bytes(dtype);
  const size_t nx = (size_t)M * d * e, nw = (size_t)d * d_ff * e, nh = (size_t)M * d_ff * e;
  if ((nx && !x) || (nw && (!wg || !wu)) || (nh && !h))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((x && !aligned16(x)) || (wg && !aligned16(wg)) || (wu && !aligned16(wu)) || (h && !aligned16(h)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(h, nh, x, nx) || overlaps(h, nh, wg, nw) || overlaps(h, nh, wu, nw))
    return fail(SWIGLU_ERR_INVALID_ARG, "h overlaps an input");
  return SWIGLU_OK;
}

// y [M, d] = h [M, d_ff] . W_down [d_ff, d] (+ r [M, d]); r may be y itself.
int validate_down(const void* h, const void* wd, const void* r, const void* y, int64_t M,
                  int64_t d_ff, int64_t d, int dtype) {
  int v = check_sizes(M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  const size_t e = (size_t)elem_bytes(dtype);
  const size_t nh = (size_t)M * d_ff * e, nw = (size_t)d_ff * d * e, ny = (size_t)M * d * e;
  if ((nh && !h) || (nw && !wd) || (ny && !y))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((h && !aligned16(h)) || (wd && !aligned16(wd)) || (r && !aligned16(r)) ||
      (y && !aligned16(y)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(y, ny, h, nh) || overlaps(y, ny, wd, nw))
    return fail(SWIGLU_ERR_INVALID_ARG, "y overlaps an input");
  if (r && r != y && overlaps(y, ny, r, ny))
    return fail(SWIGLU_ERR_INVALID_ARG, "residual partially overlaps y");
  return SWIGLU_OK;
}

struct Plan {
  int path;
  SimtPlan simt;
  SkinnyPlan skinny;
  TilePlan tile;
  int64_t slices;
  int64_t grid;
  int64_t launches;   // kernels one call launches
  int64_t cluster;    // CTAs per cluster of the main kernel (1 = none)
  size_t workspace;
  bool inject_oom;    // the SWIGLU_INJECT_OOM test hook is set
};

// K: shared dimension; n_out: output columns (up: d, d_ff; down: d_ff, d).
// max_pairs: 2-CTA clusters that fit on the device at once (num_sms / 2 when
// planning without a device).
// nk: the weights are [n_out, K] (served by the tensor-core paths only).
int make_plan(int op, int64_t M, int64_t K, int64_t n_out, int dtype, int path, int num_sms,
              int max_pairs, Plan* p, bool fp8 = false, const int* sk_caps = nullptr,
              bool nk = false, const int* simt_caps = nullptr) {
  int rp = 0;
  int st = resolve_path(op, M, K, n_out, dtype, path, &rp, num_sms, sk_caps);
  if (st != SWIGLU_OK) return st;
  const Tuning tn = read_tuning();
  // AUTO, bf16, one row on small weights: the SIMT path's cluster form
  // (measured, graph replay, against the skinny tcgen05 kernel: d = 512 /
  // 896 / 1024 at M = 1: 3.2 / 6.6 / 4.6 us against 4.2 / 7.0 / 6.4 us; at
  // d = 2048 it trails, 10.2 against 9.8 us).
  if (path == SWIGLU_PATH_AUTO && op == kOpUp && dtype == SWIGLU_BF16 && !fp8 && !nk &&
      simt_cluster_plan(M, K, n_out, dtype, tn, simt_caps) && K <= kSimtClusterPreferMaxK)
    rp = SWIGLU_PATH_SIMT;
  *p = Plan{};
  p->path = rp;
  p->cluster = 1;
  const bool plain = op == kOpDown;
  p->inject_oom = tn.inject_oom != 0;
  if (rp == SWIGLU_PATH_SIMT) {
    p->simt = plan_simt(M, K, n_out, dtype, num_sms, tn);
    if (p->simt.slices > kMaxGridYZ || p->simt.row_chunks > kMaxGridYZ)
      return fail(SWIGLU_ERR_UNSUPPORTED, "shape exceeds the grid limits of the SIMT path");
    p->simt.cluster = simt_cluster_plan(M, K, n_out, dtype, tn, simt_caps);
    if (p->simt.cluster) {
      // one launch: K slices in clusters of CTAs, no workspace
      const int64_t cols = dtype == SWIGLU_BF16 ? 64 : 32;
      p->simt.fused = false;
      p->simt.counters_bytes = 0;
      p->slices = p->simt.cluster;
      p->grid = (n_out + cols - 1) / cols * p->slices;
      p->workspace = 0;
      p->launches = 1;
      p->cluster = p->simt.cluster;
    } else {
      p->slices = p->simt.slices;
      p->grid = p->simt.col_blocks * p->simt.slices * p->simt.row_chunks;
      p->workspace = p->simt.counters_bytes + partial_elems(p->slices, M, n_out) * sizeof(float);
      p->launches = p->slices > 0 && !p->simt.fused ? 2 : 1;
    }
  } else if (rp == SWIGLU_PATH_SKINNY) {
    p->skinny = plan_skinny(M, K, n_out, num_sms, plain, fp8, sk_caps, tn);
    // K slices per column group: the cluster size, or (stream-K) at most maxq
    p->slices = p->skinny.cluster ? p->skinny.cluster : p->skinny.maxq;
    p->grid = p->skinny.grid;
    p->workspace = p->skinny.counters_bytes + p->skinny.part_bytes;
    p->launches = p->skinny.split ? 2 : 1;
    p->cluster = p->skinny.cluster ? p->skinny.cluster : 1;
  } else {
    p->tile = plan_tile(M, K, n_out, num_sms, plain, max_pairs, tn);
    p->slices = 1;
    p->grid = p->tile.grid;
    p->workspace = p->tile.counters_bytes + p->tile.part_bytes;
    p->launches = 1;
    p->cluster = p->tile.pair ? 2 : 1;
  }
  if (M == 0 || n_out == 0) p->launches = 0;
  if (plain && K == 0) p->launches = 0;
  p->workspace = (p->workspace + 255) / 256 * 256;
  return SWIGLU_OK;
}

// One call of either operation: x [M, K] times the weights, into out [M, n_out].
struct Call {
  int op;
  const void *x, *wa, *wb, *resid;
  void* out;
  int64_t M, K, n_out;
  int dtype, path;
  void* workspace;
  size_t ws_bytes;
  cudaStream_t st;
  int wlayout;   // a WeightLayout: [K, n_out], [n_out, K] (torch.nn.Linear.weight) or packed
  // FP8 up projection: x is bf16 and is quantized per row to e4m3 in the
  // workspace; wa, wb are e4m3 codes [n_out, K] with column scales sw_a, sw_b.
  bool fp8 = false;
  const float* sw_a = nullptr;
  const float* sw_b = nullptr;
};

// Bytes an FP8 call keeps ahead of its partial sums: x's codes and row scales.
size_t fp8_prefix_bytes(int64_t M, int64_t K) {
  return ((size_t)M * K + 255) / 256 * 256 + ((size_t)M * 4 + 255) / 256 * 256;
}

int run(const Call& c) {
  int v;
  int dev = 0;
  DeviceInfo di;
  if ((v = current_device(&dev, &di)) != SWIGLU_OK) return v;
  Plan p;
  // FP8: the GEMM kernels see each row of e4m3 codes as K / 2 byte pairs
  const int64_t Kg = c.fp8 ? c.K / 2 : c.K;
  if ((v = make_plan(c.op, c.M, Kg, c.n_out, c.dtype, c.path, di.num_sms, di.max_pairs, &p,
                     c.fp8, di.sk_caps, c.wlayout == kWeightsNK, di.simt_caps)) != SWIGLU_OK)
    return v;
  if (c.fp8 && p.path == SWIGLU_PATH_SIMT && c.K > 0)
    return fail(SWIGLU_ERR_UNSUPPORTED, "FP8 weights are served by the tensor-core paths only");
  const size_t fp8_prefix = c.fp8 && p.path != SWIGLU_PATH_SIMT ? fp8_prefix_bytes(c.M, c.K) : 0;
  p.workspace += fp8_prefix;
  if (c.wlayout == kWeightsNK && p.path == SWIGLU_PATH_SIMT && c.K > 0)
    return fail(SWIGLU_ERR_UNSUPPORTED,
                "[N, K] weights are served by the tensor-core paths (bf16) only");
  if (p.path == SWIGLU_PATH_SIMT && p.simt.fused) {
    // Inside a CUDA graph the two-launch form is kept: it needs no arrival
    // counters.  (It was chosen when a captured call's workspace needed a
    // memset node; the zeroed slices of graph_workspace have not been
    // measured with the single launch.)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(c.st, &cs) != cudaSuccess) {
      cudaGetLastError();
    } else if (cs != cudaStreamCaptureStatusNone) {
      p.simt.fused = false;
      p.simt.counters_bytes = 0;
      p.workspace = (partial_elems(p.slices, c.M, c.n_out) * sizeof(float) + 255) / 256 * 256;
      p.launches = 2;
    }
  }
  if (c.M == 0 || c.n_out == 0) {
    t_err[0] = 0;
    return SWIGLU_OK;
  }
  const size_t out_bytes = (size_t)c.M * c.n_out * elem_bytes(c.dtype);
  if (c.op == kOpDown && c.K == 0) {
    // empty sums: y = residual, or 0
    cudaError_t e = c.resid ? (c.resid == c.out ? cudaSuccess
                                                : cudaMemcpyAsync(c.out, c.resid, out_bytes,
                                                                  cudaMemcpyDeviceToDevice, c.st))
                            : cudaMemsetAsync(c.out, 0, out_bytes, c.st);
    if (e != cudaSuccess) return cuda_fail(e, "empty-sum fill");
    t_err[0] = 0;
    return SWIGLU_OK;
  }
  if (c.workspace && overlaps(c.out, out_bytes, c.workspace, c.ws_bytes))
    return fail(SWIGLU_ERR_INVALID_ARG, "the output overlaps the workspace");

  // Where the partial sums (and the arrival counters) live:
  //   caller workspace -> [counters][partials] inside it, counters cleared;
  //   else the stream's cached buffer -> counters already zero;
  //   else a per-call pool allocation -> counters cleared.
  // An FP8 call keeps x's codes and row scales ahead of them: at the start
  // of a caller workspace (a documented layout), else at the start of the
  // partial-sum region.
  char* fp8_base = nullptr;
  float* part = nullptr;
  unsigned* counters = nullptr;
  bool counters_clean = false;
  void* pooled = nullptr;
  const size_t counter_bytes = p.path == SWIGLU_PATH_SKINNY ? p.skinny.counters_bytes
                               : p.path == SWIGLU_PATH_TC   ? p.tile.counters_bytes
                                                            : p.simt.counters_bytes;
  cudaStream_t st = c.st;
  if (p.workspace > 0) {
    if (c.workspace) {
      if (c.ws_bytes < p.workspace || ((uintptr_t)c.workspace & 255u))
        return fail(SWIGLU_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)",
                    p.workspace, c.ws_bytes);
      fp8_base = (char*)c.workspace;
      counters = (unsigned*)((char*)c.workspace + fp8_prefix);
      part = (float*)((char*)c.workspace + fp8_prefix + counter_bytes);
    } else {
      if (!p.inject_oom &&
          (v = stream_workspace(dev, st, p.workspace - counter_bytes, &part, &counters)) != SWIGLU_OK)
        return v;
      if (part) {
        counters_clean = true;
        fp8_base = (char*)part;
        part = (float*)((char*)part + fp8_prefix);
        if (counter_bytes) ensure_graph_counters(dev, st);
      } else if (char* gw = p.inject_oom ? nullptr : graph_workspace(dev, st, p.workspace)) {
        // a captured call: its capture's slice (see GraphSlice), counters clean
        counters = (unsigned*)gw;
        counters_clean = true;
        fp8_base = gw + counter_bytes;
        part = (float*)(fp8_base + fp8_prefix);
      } else {
        // A captured call takes clean counters from the graph-counter region
        // when it can (see GraphCounters) and allocates only the rest.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (counter_bytes && !p.inject_oom && cudaStreamIsCapturing(st, &cs) == cudaSuccess &&
            cs != cudaStreamCaptureStatusNone)
          counters = take_graph_counters(dev, counter_bytes);
        cudaGetLastError();
        const size_t own = counters ? p.workspace - counter_bytes : p.workspace;
        if (own > 0 && p.inject_oom)
          return fail(SWIGLU_ERR_OOM, "workspace of %zu bytes: allocation failure injected "
                      "(SWIGLU_INJECT_OOM)", own);
        if (own > 0) {
          cudaMemPool_t pool;
          if ((v = device_pool(dev, &pool)) != SWIGLU_OK) return v;
          cudaError_t e = cudaMallocFromPoolAsync(&pooled, own, pool, st);
          if (e != cudaSuccess) {
            if (e == cudaErrorMemoryAllocation) {
              cudaGetLastError();
              return fail(SWIGLU_ERR_OOM, "workspace of %zu bytes: %s", own,
                          cudaGetErrorString(e));
            }
            return cuda_fail(e, "cudaMallocFromPoolAsync");
          }
        }
        if (counters) {
          counters_clean = true;
          fp8_base = (char*)pooled;
        } else {
          counters = (unsigned*)pooled;
          fp8_base = (char*)pooled + counter_bytes;
        }
        part = (float*)(fp8_base + fp8_prefix);
      }
    }
  }

  cudaError_t e = cudaSuccess;
  const void* xg = c.x;   // what the GEMM kernels read as x
  Fp8Scales fs{nullptr, c.sw_a, c.sw_b};
  if (fp8_prefix) {
    uint8_t* x8 = (uint8_t*)fp8_base;
    float* sx = (float*)(x8 + ((size_t)c.M * c.K + 255) / 256 * 256);
    e = launch_quantize_rows_fp8(c.x, x8, sx, c.M, c.K, st);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    xg = x8;
    fs.sx = sx;
  }
  const Fp8Scales* fsp = fp8_prefix ? &fs : nullptr;
  if (p.path == SWIGLU_PATH_SIMT && p.simt.cluster) {
    e = launch_simt_cluster(c.x, c.wa, c.wb, c.out, c.M, c.K, c.n_out, c.dtype, p.simt.cluster,
                            c.wlayout == kWeightsPacked, st);
  } else if (p.path == SWIGLU_PATH_SIMT && p.simt.fused) {
    e = launch_simt_partial(c.x, c.wa, c.wb, part, c.M, c.K, c.n_out, c.dtype, p.simt, st,
                            counters, counters_clean, c.out, c.wlayout == kWeightsPacked);
  } else if (p.path == SWIGLU_PATH_SIMT) {
    e = launch_simt_partial(c.x, c.wa, c.wb, part, c.M, c.K, c.n_out, c.dtype, p.simt, st,
                            nullptr, false, nullptr, c.wlayout == kWeightsPacked);
    if (e == cudaSuccess)
      e = launch_reduce_swiglu(part, c.out, c.M, c.n_out, p.slices, c.dtype, di.num_sms, st);
  } else if (p.path == SWIGLU_PATH_SKINNY) {
    e = launch_skinny_tc(xg, c.wa, c.wb, c.out, c.resid, c.M, Kg, c.n_out, c.wlayout, p.skinny,
                         part, counters, counters_clean, di.status, wait_timeout_ns(), st, fsp);
  } else {
    e = launch_tile_tc(xg, c.wa, c.wb, c.out, c.resid, c.M, Kg, c.n_out, c.wlayout, p.tile,
                       part, counters, counters_clean, di.status, wait_timeout_ns(), st, fsp);
  }
  if (pooled) {
    cudaError_t ef = cudaFreeAsync(pooled, st);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  t_err[0] = 0;
  return SWIGLU_OK;
}

int run_up(const void* x, const void* wg, const void* wu, void* h, int64_t M, int64_t d,
           int64_t d_ff, int dtype, int path, void* workspace, size_t ws_bytes,
           cudaStream_t st, int wlayout = kWeightsKN) {
  int v = validate(x, wg, wu, h, M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  return run(Call{kOpUp, x, wg, wu, nullptr, h, M, d, d_ff, dtype, path, workspace, ws_bytes, st,
                  wlayout});
}

// x [M, d], w_packed [d, packed_cols(d_ff)] (launch_pack's layout), h [M, d_ff].
int validate_packed(const void* x, const void* wp, const void* h, int64_t M, int64_t d,
                    int64_t d_ff, int dtype) {
  int v = check_sizes(M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  const size_t e = (size_t)elem_bytes(dtype);
  const size_t nx = (size_t)M * d * e, nw = (size_t)d * packed_cols(d_ff) * e;
  const size_t nh = (size_t)M * d_ff * e;
  if ((nx && !x) || (nw && !wp) || (nh && !h))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((x && !aligned16(x)) || (wp && !aligned16(wp)) || (h && !aligned16(h)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(h, nh, x, nx) || overlaps(h, nh, wp, nw))
    return fail(SWIGLU_ERR_INVALID_ARG, "h overlaps an input");
  return SWIGLU_OK;
}

// x [M, d] bf16, w8 [d_ff, d] e4m3 codes (x2), scales [d_ff] f32 (x2), h [M, d_ff] bf16.
int validate_fp8(const void* x, const void* w8g, const void* w8u, const float* sg,
                 const float* su, const void* h, int64_t M, int64_t d, int64_t d_ff) {
  int v = check_sizes(M, d, d_ff, SWIGLU_BF16);
  if (v != SWIGLU_OK) return v;
  if (d % 16 != 0)
    return fail(SWIGLU_ERR_ALIGNMENT, "d must be a multiple of 16 for e4m3 rows");
  const size_t nx = (size_t)M * d * 2, nw = (size_t)d * d_ff, ns = (size_t)d_ff * 4;
  const size_t nh = (size_t)M * d_ff * 2;
  if ((nx && !x) || (nw && (!w8g || !w8u || !sg || !su)) || (nh && !h))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((x && !aligned16(x)) || (w8g && !aligned16(w8g)) || (w8u && !aligned16(w8u)) ||
      (sg && !aligned16(sg)) || (su && !aligned16(su)) || (h && !aligned16(h)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(h, nh, x, nx) || overlaps(h, nh, w8g, nw) || overlaps(h, nh, w8u, nw) ||
      overlaps(h, nh, sg, ns) || overlaps(h, nh, su, ns))
    return fail(SWIGLU_ERR_INVALID_ARG, "h overlaps an input");
  return SWIGLU_OK;
}

int run_down(const void* h, const void* wd, const void* r, void* y, int64_t M, int64_t d_ff,
             int64_t d, int dtype, int path, void* workspace, size_t ws_bytes,
             cudaStream_t st, int wlayout = kWeightsKN) {
  int v = validate_down(h, wd, r, y, M, d_ff, d, dtype);
  if (v != SWIGLU_OK) return v;
  return run(Call{kOpDown, h, wd, wd, r, y, M, d_ff, d, dtype, path, workspace, ws_bytes, st,
                  wlayout});
}

}  // namespace

int64_t split_k_slices(int64_t K, int64_t col_blocks, int64_t target_blocks,
                       int64_t min_k_per_slice) {
  if (K < 0 || col_blocks <= 0 || target_blocks <= 0 || min_k_per_slice <= 0) return -1;
  int64_t want = (target_blocks + col_blocks - 1) / col_blocks;   // slices to reach the target
  int64_t most = K / min_k_per_slice;                              // keep >= min_k per slice
  if (most < 1) most = 1;
  if (want > most) want = most;
  if (want < 1) want = 1;
  return want;
}

int api_validate(const void* x, const void* wg, const void* wu, const void* h, int64_t M,
                 int64_t d, int64_t d_ff, int dtype) {
  return validate(x, wg, wu, h, M, d, d_ff, dtype);
}

int api_current_device(int* dev, int* num_sms) {
  DeviceInfo di;
  int v = current_device(dev, &di);
  if (v == SWIGLU_OK) *num_sms = di.num_sms;
  return v;
}

int api_fail(int status, const char* detail) { return fail(status, "%s", detail); }

int api_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }

void api_clear_error() { t_err[0] = 0; }

unsigned* api_status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_dev[dev].status;
}

}  // namespace swg

using namespace swg;

extern "C" {

int swiglu_up(const void* x, const void* w_gate, const void* w_up, void* h,
              int64_t M, int64_t d, int64_t d_ff, int dtype, void* stream) {
  return run_up(x, w_gate, w_up, h, M, d, d_ff, dtype, SWIGLU_PATH_AUTO, nullptr, 0,
                (cudaStream_t)stream);
}

int swiglu_up_ex(const void* x, const void* w_gate, const void* w_up, void* h,
                 int64_t M, int64_t d, int64_t d_ff, int dtype, int path,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return run_up(x, w_gate, w_up, h, M, d, d_ff, dtype, path, workspace, workspace_bytes,
                (cudaStream_t)stream);
}

int swiglu_down(const void* h, const void* w_down, const void* residual, void* y, int64_t M,
                int64_t d_ff, int64_t d, int dtype, void* stream) {
  return run_down(h, w_down, residual, y, M, d_ff, d, dtype, SWIGLU_PATH_AUTO, nullptr, 0,
                  (cudaStream_t)stream);
}

int swiglu_down_ex(const void* h, const void* w_down, const void* residual, void* y,
                   int64_t M, int64_t d_ff, int64_t d, int dtype, int path, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return run_down(h, w_down, residual, y, M, d_ff, d, dtype, path, workspace, workspace_bytes,
                  (cudaStream_t)stream);
}

int swiglu_up_nk(const void* x, const void* w_gate_nk, const void* w_up_nk, void* h, int64_t M,
                 int64_t d, int64_t d_ff, int dtype, int path, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return run_up(x, w_gate_nk, w_up_nk, h, M, d, d_ff, dtype, path, workspace, workspace_bytes,
                (cudaStream_t)stream, kWeightsNK);
}

size_t swiglu_packed_weight_bytes(int64_t d, int64_t d_ff, int dtype) {
  if (check_sizes(0, d, d_ff, dtype) != SWIGLU_OK) return 0;
  t_err[0] = 0;
  return (size_t)d * (size_t)packed_cols(d_ff) * (size_t)elem_bytes(dtype);
}

int swiglu_pack_weights(const void* w_gate, const void* w_up, void* w_packed, int64_t d,
                        int64_t d_ff, int dtype, void* stream) {
  int v = check_sizes(0, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  const size_t e = (size_t)elem_bytes(dtype);
  const size_t nw = (size_t)d * d_ff * e, np = (size_t)d * packed_cols(d_ff) * e;
  if (nw && (!w_gate || !w_up || !w_packed))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((w_gate && !aligned16(w_gate)) || (w_up && !aligned16(w_up)) ||
      (w_packed && !aligned16(w_packed)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(w_packed, np, w_gate, nw) || overlaps(w_packed, np, w_up, nw))
    return fail(SWIGLU_ERR_INVALID_ARG, "the packed matrix overlaps an input");
  int dev = 0;
  DeviceInfo di;
  if ((v = current_device(&dev, &di)) != SWIGLU_OK) return v;
  if (nw == 0) {
    t_err[0] = 0;
    return SWIGLU_OK;
  }
  cudaError_t e2 = launch_pack(w_gate, w_up, w_packed, d, d_ff, dtype, di.num_sms,
                               (cudaStream_t)stream);
  if (e2 != cudaSuccess) return cuda_fail(e2, "kernel launch");
  t_err[0] = 0;
  return SWIGLU_OK;
}

// The weight quantizers: `n` bf16 matrices w[i] [K, N] row-major -> e4m3
// codes w8[i] [N, K] and f32 column scales s[i] [N], all checked first (sizes,
// null pointers, 16-byte alignment, no output overlapping an input or another
// output), with one short-lived N * 4-byte pool allocation for the column
// maxima.
static int quantize_weights(int n, const void* const* w, void* const* w8, float* const* s,
                            int64_t K, int64_t N, const char* kname, cudaStream_t st) {
  int v = check_sizes(0, K, N, SWIGLU_BF16);
  if (v != SWIGLU_OK) return v;
  if (K % 16 != 0)
    return fail(SWIGLU_ERR_ALIGNMENT, "%s must be a multiple of 16 for e4m3 rows", kname);
  const size_t nw = (size_t)K * N * 2, n8 = (size_t)K * N, ns = (size_t)N * 4;
  const void* outs[4];
  size_t out_n[4];
  for (int i = 0; i < n; ++i) {
    if (n8 && (!w[i] || !w8[i] || !s[i]))
      return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
    if ((w[i] && !aligned16(w[i])) || (w8[i] && !aligned16(w8[i])) || (s[i] && !aligned16(s[i])))
      return fail(SWIGLU_ERR_ALIGNMENT, "pointers must be 16-byte aligned");
    outs[2 * i] = w8[i];
    out_n[2 * i] = n8;
    outs[2 * i + 1] = s[i];
    out_n[2 * i + 1] = ns;
  }
  for (int i = 0; i < 2 * n; ++i) {
    for (int j = 0; j < n; ++j)
      if (overlaps(outs[i], out_n[i], w[j], nw))
        return fail(SWIGLU_ERR_INVALID_ARG, "an output overlaps an input");
    for (int j = 0; j < i; ++j)
      if (overlaps(outs[i], out_n[i], outs[j], out_n[j]))
        return fail(SWIGLU_ERR_INVALID_ARG, "outputs overlap");
  }
  int dev = 0;
  DeviceInfo di;
  if ((v = current_device(&dev, &di)) != SWIGLU_OK) return v;
  if (n8 == 0) {
    t_err[0] = 0;
    return SWIGLU_OK;
  }
  cudaMemPool_t pool;
  if ((v = device_pool(dev, &pool)) != SWIGLU_OK) return v;
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, (size_t)N * sizeof(unsigned), pool, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SWIGLU_ERR_OOM, "column maxima: %s", cudaGetErrorString(e));
  }
  for (int i = 0; i < n && e == cudaSuccess; ++i)
    e = launch_quantize_cols_fp8(w[i], w8[i], s[i], (unsigned*)scratch, K, N, di.num_sms, st);
  const cudaError_t ef = cudaFreeAsync(scratch, st);
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  t_err[0] = 0;
  return SWIGLU_OK;
}

int swiglu_quantize_weights_fp8(const void* w_gate, const void* w_up, void* w8_gate,
                                void* w8_up, float* s_gate, float* s_up, int64_t d,
                                int64_t d_ff, void* stream) {
  const void* w[2] = {w_gate, w_up};
  void* w8[2] = {w8_gate, w8_up};
  float* s[2] = {s_gate, s_up};
  return quantize_weights(2, w, w8, s, d, d_ff, "d", (cudaStream_t)stream);
}

int swiglu_quantize_weight_fp8(const void* w, void* w8, float* s, int64_t K, int64_t N,
                               void* stream) {
  return quantize_weights(1, &w, &w8, &s, K, N, "K", (cudaStream_t)stream);
}

int swiglu_down_fp8(const void* h, const void* w8_down, const float* s_down,
                    const void* residual, void* y, int64_t M, int64_t d_ff, int64_t d, int path,
                    void* workspace, size_t workspace_bytes, void* stream) {
  // As validate_down, with 1-byte weight codes and the scale vector.
  int v = check_sizes(M, d, d_ff, SWIGLU_BF16);
  if (v != SWIGLU_OK) return v;
  if (d_ff % 16 != 0)
    return fail(SWIGLU_ERR_ALIGNMENT, "d_ff must be a multiple of 16 for e4m3 rows");
  const size_t nh = (size_t)M * d_ff * 2, nw = (size_t)d_ff * d, ns = (size_t)d * 4;
  const size_t ny = (size_t)M * d * 2;
  if ((nh && !h) || (nw && (!w8_down || !s_down)) || (ny && !y))
    return fail(SWIGLU_ERR_INVALID_ARG, "null pointer for a non-empty tensor");
  if ((h && !aligned16(h)) || (w8_down && !aligned16(w8_down)) || (s_down && !aligned16(s_down)) ||
      (residual && !aligned16(residual)) || (y && !aligned16(y)))
    return fail(SWIGLU_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if (overlaps(y, ny, h, nh) || overlaps(y, ny, w8_down, nw) || overlaps(y, ny, s_down, ns))
    return fail(SWIGLU_ERR_INVALID_ARG, "y overlaps an input");
  if (residual && residual != y && overlaps(y, ny, residual, ny))
    return fail(SWIGLU_ERR_INVALID_ARG, "residual partially overlaps y");
  Call c{kOpDown, h, w8_down, w8_down, residual, y, M, d_ff, d, SWIGLU_BF16, path, workspace,
         workspace_bytes, (cudaStream_t)stream, kWeightsNK};
  c.fp8 = true;
  c.sw_a = s_down;
  c.sw_b = s_down;
  return run(c);
}

size_t swiglu_down_fp8_workspace_bytes(int64_t M, int64_t d_ff, int64_t d, int path) {
  if (check_sizes(M < 0 ? -1 : M, d, d_ff, SWIGLU_BF16) != SWIGLU_OK) return 0;
  if (d_ff % 16 != 0) {
    fail(SWIGLU_ERR_ALIGNMENT, "d_ff must be a multiple of 16 for e4m3 rows");
    return 0;
  }
  int dev = 0;
  DeviceInfo di;
  if (current_device(&dev, &di) != SWIGLU_OK) return 0;
  Plan p;
  if (make_plan(kOpDown, M, d_ff / 2, d, SWIGLU_BF16, path, di.num_sms, di.max_pairs, &p, true,
                di.sk_caps) != SWIGLU_OK)
    return 0;
  t_err[0] = 0;
  return p.workspace + fp8_prefix_bytes(M, d_ff);
}

int swiglu_up_fp8(const void* x, const void* w8_gate, const void* w8_up, const float* s_gate,
                  const float* s_up, void* h, int64_t M, int64_t d, int64_t d_ff, int path,
                  void* workspace, size_t workspace_bytes, void* stream) {
  int v = validate_fp8(x, w8_gate, w8_up, s_gate, s_up, h, M, d, d_ff);
  if (v != SWIGLU_OK) return v;
  Call c{kOpUp, x, w8_gate, w8_up, nullptr, h, M, d, d_ff, SWIGLU_BF16, path, workspace,
         workspace_bytes, (cudaStream_t)stream, kWeightsNK};
  c.fp8 = true;
  c.sw_a = s_gate;
  c.sw_b = s_up;
  return run(c);
}

size_t swiglu_fp8_workspace_bytes(int64_t M, int64_t d, int64_t d_ff, int path) {
  if (check_sizes(M < 0 ? -1 : M, d, d_ff, SWIGLU_BF16) != SWIGLU_OK) return 0;
  if (d % 16 != 0) {
    fail(SWIGLU_ERR_ALIGNMENT, "d must be a multiple of 16 for e4m3 rows");
    return 0;
  }
  int dev = 0;
  DeviceInfo di;
  if (current_device(&dev, &di) != SWIGLU_OK) return 0;
  Plan p;
  if (make_plan(kOpUp, M, d / 2, d_ff, SWIGLU_BF16, path, di.num_sms, di.max_pairs, &p, true,
                di.sk_caps) != SWIGLU_OK)
    return 0;
  if (p.path == SWIGLU_PATH_SIMT && d > 0) {
    fail(SWIGLU_ERR_UNSUPPORTED, "FP8 weights are served by the tensor-core paths only");
    return 0;
  }
  t_err[0] = 0;
  return p.workspace + (p.path != SWIGLU_PATH_SIMT ? fp8_prefix_bytes(M, d) : 0);
}

int swiglu_up_packed(const void* x, const void* w_packed, void* h, int64_t M, int64_t d,
                     int64_t d_ff, int dtype, int path, void* workspace,
                     size_t workspace_bytes, void* stream) {
  int v = validate_packed(x, w_packed, h, M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  return run(Call{kOpUp, x, w_packed, w_packed, nullptr, h, M, d, d_ff, dtype, path, workspace,
                  workspace_bytes, (cudaStream_t)stream, kWeightsPacked});
}

int swiglu_down_nk(const void* h, const void* w_down_nk, const void* residual, void* y,
                   int64_t M, int64_t d_ff, int64_t d, int dtype, int path, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return run_down(h, w_down_nk, residual, y, M, d_ff, d, dtype, path, workspace,
                  workspace_bytes, (cudaStream_t)stream, kWeightsNK);
}

int swiglu_mlp(const void* x, const void* w_gate, const void* w_up, const void* w_down,
               const void* residual, void* h, void* y, int64_t M, int64_t d, int64_t d_ff,
               int dtype, void* stream) {
  // Both steps are validated before either is enqueued.
  int v = validate(x, w_gate, w_up, h, M, d, d_ff, dtype);
  if (v != SWIGLU_OK) return v;
  if ((v = validate_down(h, w_down, residual, y, M, d_ff, d, dtype)) != SWIGLU_OK) return v;
  if (dtype != SWIGLU_BF16)
    return fail(SWIGLU_ERR_UNSUPPORTED, "the down projection serves bf16 only");
  const size_t e = (size_t)elem_bytes(dtype);
  if (overlaps(y, (size_t)M * d * e, x, (size_t)M * d * e) && y != x)
    return fail(SWIGLU_ERR_INVALID_ARG, "y partially overlaps x");
  if (y == x && residual != x)
    return fail(SWIGLU_ERR_INVALID_ARG, "y may alias x only when x is also the residual");
  v = run_up(x, w_gate, w_up, h, M, d, d_ff, dtype, SWIGLU_PATH_AUTO, nullptr, 0,
             (cudaStream_t)stream);
  if (v != SWIGLU_OK) return v;
  return run_down(h, w_down, residual, y, M, d_ff, d, dtype, SWIGLU_PATH_AUTO, nullptr, 0,
                  (cudaStream_t)stream);
}

size_t swiglu_workspace_bytes(int64_t M, int64_t d, int64_t d_ff, int dtype, int path) {
  if (check_sizes(M < 0 ? -1 : M, d, d_ff, dtype) != SWIGLU_OK) return 0;
  int dev = 0;
  DeviceInfo di;
  if (current_device(&dev, &di) != SWIGLU_OK) return 0;
  Plan p;
  if (make_plan(kOpUp, M, d, d_ff, dtype, path, di.num_sms, di.max_pairs, &p, false,
                di.sk_caps, false, di.simt_caps) != SWIGLU_OK)
    return 0;
  return p.workspace;
}

size_t swiglu_down_workspace_bytes(int64_t M, int64_t d_ff, int64_t d, int dtype, int path) {
  if (check_sizes(M < 0 ? -1 : M, d, d_ff, dtype) != SWIGLU_OK) return 0;
  int dev = 0;
  DeviceInfo di;
  if (current_device(&dev, &di) != SWIGLU_OK) return 0;
  Plan p;
  if (make_plan(kOpDown, M, d_ff, d, dtype, path, di.num_sms, di.max_pairs, &p, false,
                di.sk_caps) != SWIGLU_OK)
    return 0;
  return p.workspace;
}

// num_sms > 0: host-only, for a device with that many SMs (cluster
// capacities estimated from it).  num_sms == 0: the current device, with the
// SM count and cluster capacities a call would use.
static int plan_common(int op, int64_t M, int64_t K, int64_t n_out, int dtype, int path,
                       int num_sms, swiglu_plan_info* out) {
  if (!out) return fail(SWIGLU_ERR_INVALID_ARG, "null output");
  if (dtype != SWIGLU_F32 && dtype != SWIGLU_BF16) return fail(SWIGLU_ERR_INVALID_ARG, "unknown dtype %d", dtype);
  if (M < 0 || K < 0 || n_out < 0 || num_sms < 0) return fail(SWIGLU_ERR_INVALID_ARG, "negative size or SM count");
  Plan p;
  int v;
  const int* sk_caps = nullptr;
  DeviceInfo di;
  if (num_sms == 0) {
    int dev = 0;
    if ((v = current_device(&dev, &di)) != SWIGLU_OK) return v;
    num_sms = di.num_sms;
    sk_caps = di.sk_caps;
    v = make_plan(op, M, K, n_out, dtype, path, di.num_sms, di.max_pairs, &p, false, sk_caps,
                  false, di.simt_caps);
  } else {
    v = make_plan(op, M, K, n_out, dtype, path, num_sms, num_sms / 2, &p);
  }
  if (v != SWIGLU_OK) return v;
  out->path = p.path;
  out->slices = p.slices;
  out->grid = p.grid;
  out->row_chunk = p.path == SWIGLU_PATH_SIMT ? p.simt.row_chunk : 0;
  out->workspace = (int64_t)p.workspace;
  out->skinny_max_m = skinny_max_m(op, K, n_out, num_sms, sk_caps);
  out->launches = p.launches;
  out->cluster = p.cluster;
  return SWIGLU_OK;
}

int swiglu_plan(int64_t M, int64_t d, int64_t d_ff, int dtype, int path, int num_sms,
                swiglu_plan_info* out) {
  return plan_common(kOpUp, M, d, d_ff, dtype, path, num_sms, out);
}

int swiglu_down_plan(int64_t M, int64_t d_ff, int64_t d, int dtype, int path, int num_sms,
                     swiglu_plan_info* out) {
  return plan_common(kOpDown, M, d_ff, d, dtype, path, num_sms, out);
}

int64_t swiglu_split_k_slices(int64_t K, int64_t col_blocks, int64_t target_blocks,
                              int64_t min_k_per_slice) {
  return split_k_slices(K, col_blocks, target_blocks, min_k_per_slice);
}

int swiglu_check_device_status(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_status, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  if (word) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) mark_workspaces_dirty(dev);
    return fail(SWIGLU_ERR_TIMEOUT,
                "a device-side wait gave up, found a stale arrival counter or a CTA pair's "
                "TMEM allocations disagreed (status word 0x%x)",
                word);
  }
  return SWIGLU_OK;
}

int swiglu_release_stream_workspace(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int v = release_stream_workspace(dev, (cudaStream_t)stream);
  if (v == SWIGLU_OK) t_err[0] = 0;
  return v;
}

int swiglu_release_workspaces(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int v = release_device_workspaces(dev);
  if (v == SWIGLU_OK) t_err[0] = 0;
  return v;
}

size_t swiglu_cached_workspace_bytes(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 0;
  }
  return cached_workspace_bytes(dev);
}

const char* swiglu_status_string(int status) {
  switch (status) {
    case SWIGLU_OK: return "ok";
    case SWIGLU_ERR_INVALID_ARG: return "invalid argument";
    case SWIGLU_ERR_UNSUPPORTED: return "unsupported";
    case SWIGLU_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case SWIGLU_ERR_OOM: return "out of device memory";
    case SWIGLU_ERR_CUDA: return "CUDA error";
    case SWIGLU_ERR_TIMEOUT: return "device-side wait timed out";
    case SWIGLU_ERR_ARCH: return "device is not sm_103";
    case SWIGLU_ERR_WORKSPACE: return "workspace too small or misaligned";
    default: return "unknown status";
  }
}

const char* swiglu_last_error_string(void) { return t_err; }

int swiglu_version(void) { return 200; }

}  // extern "C"
