// gda_api.cu -- the C ABI of include/gda.h: validation, workspace, planning, launches.
//
// Host-side checks run before any CUDA call (so they work without a GPU); nothing
// is read back from the device on the decode path (gda_decode_step_host's copy of its
// result to host memory aside).  gda_decode keeps one workspace
// per device and grows it with cudaMalloc (never while the stream is capturing);
// gda_decode_ex takes the caller's workspace and allocates nothing (cuDNN FE-OSS
// "Gated Attention Block (SM107)", Forward: execute() allocates nothing and is
// CUDA-graph friendly; FreeToken PR #781, Summary: initialise before capture,
// validate before launch).
#include <math.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "gda.h"
#include "gda_device.cuh"
#include "gda_kernels.h"
#include "gda_prefill.h"
#include "gda_small.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultMinChunk = 64;

struct DeviceState {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int sms = 0;
  // Buffers the internal workspace outgrew.  They are never freed: a CUDA graph
  // captured while one of them was current still reads and writes it on replay.
  std::vector<void*> retired;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Pipeline wait limit in SM cycles for later launches (0: gda::kWaitLimitCycles);
// gda_debug_wait_limit sets it for the failure-path test.
std::atomic<long long> g_wait_limit{0};

long long wait_limit() {
  const long long w = g_wait_limit.load();
  return w > 0 ? w : gda::kWaitLimitCycles;
}

// stage-1 timing (gda_timing_begin / gda_timing_end)
std::vector<cudaEvent_t> g_tev;   // pairs: [2i] before stage 1, [2i+1] after
int g_tmax = 0, g_tused = 0;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_sizes(int B, int Hq, int Hkv, int D, int num_splits) {
  if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return GDA_ERR_SHAPE;
  if (num_splits > GDA_MAX_SPLITS) return GDA_ERR_SPLITS;
  if (D != gda::kD) return GDA_ERR_UNSUPPORTED;
  return GDA_OK;
}

// Groups of up to 8 query heads ("virtual heads") each make one pass over their
// KV head's rows: G = Hq / Hkv query heads per KV head need ceil(G / 8) passes.
int passes(int Hq, int Hkv) { return (Hq / Hkv + gda::kG - 1) / gda::kG; }

size_t num_pieces(int B, int vheads, int num_splits) {
  if (num_splits > 0) return (size_t)B * vheads * num_splits;
  return (size_t)gda::kAutoMaxCtas + (size_t)B * vheads;
}

struct Layout {
  size_t o_off, lse_off, total;
};

// Groups of 8 per piece on the MMA kernel: one pass, or teams of two (2 or 4 passes)
// or three (3 or 5 and more passes: fewer reads of every row than pairs).
int team_size(int npass) { return npass <= 1 ? 1 : (npass == 2 || npass == 4) ? 2 : 3; }

// Header, then FP32 partial O [pieces][8][D], then partial LSE [pieces][8].  With two
// or more passes the size covers both schedules: per virtual head, and in teams (one
// piece per KV head and team of groups holding every group's partial), which needs
// team num_pieces(B, Hkv * ceil(passes / team)).
Layout layout(int B, int Hq, int Hkv, int D, int num_splits) {
  const int np = passes(Hq, Hkv);
  size_t pieces = num_pieces(B, Hkv * np, num_splits);
  // the BF16 kernel's team and the FP8 kernel's pairs
  const int ts[2] = {team_size(np), np >= 2 ? 2 : 1};
  for (int t : ts) {
    if (t <= 1) continue;
    const size_t pp = (size_t)t * num_pieces(B, Hkv * ((np + t - 1) / t), num_splits);
    if (pp > pieces) pieces = pp;
  }
  Layout l;
  l.o_off = gda::kHeaderBytes;
  l.lse_off = round_up(l.o_off + pieces * gda::kG * (size_t)D * sizeof(float), 256);
  l.total = round_up(l.lse_off + pieces * gda::kG * sizeof(float), 256);
  return l;
}

int sm_count(int dev) {
  if (g_dev[dev].sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
    g_dev[dev].sms = n;
  }
  return g_dev[dev].sms;
}

int validate_args(const gda_args* a) {
  if (a == nullptr) return GDA_ERR_NULL;
  int rc = check_sizes(a->B, a->Hq, a->Hkv, a->D, a->num_splits);
  if (rc != GDA_OK) return rc;
  if (a->check_indices && a->num_slots < 0) return GDA_ERR_SHAPE;
  if (a->variant < 0 || a->variant > GDA_VARIANT_TMA) return GDA_ERR_UNSUPPORTED;
  if (a->min_chunk < 0 || a->window < 0 || a->max_len < 0 || a->total_len < 0) return GDA_ERR_SHAPE;
  if (a->kv_dtype != GDA_KV_BF16 && a->kv_dtype != GDA_KV_E4M3) return GDA_ERR_UNSUPPORTED;
  if (a->kv_dtype == GDA_KV_E4M3) {
    if (a->variant != GDA_VARIANT_AUTO && a->variant != GDA_VARIANT_MMA) return GDA_ERR_UNSUPPORTED;
    if (!isfinite(a->k_descale) || !isfinite(a->v_descale)) return GDA_ERR_ARG;
  }
  if (a->B == 0) return GDA_OK;
  if (!a->q || !a->k_pool || !a->v_pool || !a->kv_indptr || !a->kv_indices || !a->out) return GDA_ERR_NULL;
  if (a->fuse_gate && !a->gate) return GDA_ERR_NULL;
  if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->v_pool, 16) || !aligned(a->out, 16) ||
      (a->gate && !aligned(a->gate, 16)) || !aligned(a->kv_indptr, 4) || !aligned(a->kv_indices, 4) ||
      (a->lse && !aligned(a->lse, 4)) || (a->sinks && !aligned(a->sinks, 4)))
    return GDA_ERR_ALIGN;
  return GDA_OK;
}

// The automatic split rule on the host: the same arithmetic as the device's
// (Sched::auto_uniform_splits) on a longest length lmax and a total n that the
// caller knows; 0 selects the stream schedule.
int host_uniform_splits(long long B, long long heads, long long grid, int min_chunk, long long lmax, long long n,
                        int kv8) {
  const long long units1 = B * heads;
  if (units1 > grid) return 0;
  if (units1 == 0) return 1;
  if (heads * n >= (long long)gda::kStreamMinPerCta * (kv8 ? 2 : 1) * grid) return 0;
  if (4 * lmax * B > 5 * n) return 0;
  long long s_opt = 1;
  const long long k = kv8 ? 16 : 4;
  while (k * s_opt * s_opt <= lmax) s_opt *= 2;
  const long long s_len = lmax > 0 ? (lmax + min_chunk - 1) / min_chunk : 1;
  long long s = s_opt < s_len ? s_opt : s_len;
  const long long s_wave = grid / units1;
  if (s >= s_wave) {
    long long p2 = 1;
    while (2 * p2 <= s_wave) p2 *= 2;
    s = (5 * p2 * units1 >= 4 * grid) ? p2 : s_wave;
    if (5 * s * units1 < 4 * grid) return 0;
  }
  return (int)s;
}

// Enqueue both stages.  Arguments validated; workspace large enough.
int enqueue(const gda_args* a, void* ws, cudaStream_t stream) {
  if (a->B == 0) return GDA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDA_ERR_CUDA;
  int sms;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    sms = sm_count(dev);
  }
  if (sms <= 0) return GDA_ERR_CUDA;

  // small batches with a host-known length bound: one cluster kernel (no partials)
  const int small_c = (a->num_splits <= 0 && a->variant == GDA_VARIANT_AUTO && !a->check_indices &&
                       a->Hq / a->Hkv <= gda::kG)
                          ? gda::small_cluster_for((long long)a->B * a->Hkv, a->max_len)
                          : 0;
  if (small_c > 0) {
    gda::SmallParams ps;
    ps.q = reinterpret_cast<const __nv_bfloat16*>(a->q);
    ps.gate = reinterpret_cast<const __nv_bfloat16*>(a->gate);
    ps.k_pool = a->k_pool;
    ps.v_pool = a->v_pool;
    ps.indptr = a->kv_indptr;
    ps.indices = a->kv_indices;
    ps.out = reinterpret_cast<__nv_bfloat16*>(a->out);
    ps.lse_out = a->lse;
    ps.sinks = a->sinks;
    ps.B = a->B;
    ps.Hq = a->Hq;
    ps.Hkv = a->Hkv;
    ps.G = a->Hq / a->Hkv;
    const bool fp8 = a->kv_dtype == GDA_KV_E4M3;
    // e4m3 pools: k_descale joins the score scale (one rounding, from double)
    ps.scale_log2 = fp8 ? (float)((double)a->scale * (double)a->k_descale * 1.4426950408889634074)
                        : a->scale * 1.44269504088896340736f;
    ps.kv_fp8 = fp8 ? 1 : 0;
    ps.v_descale = fp8 ? a->v_descale : 1.0f;
    ps.window = a->window;
    ps.fuse_gate = a->fuse_gate ? 1 : 0;
    cudaEvent_t s_end = nullptr;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if (g_tused < g_tmax) {
        if (cudaEventRecord(g_tev[2 * g_tused], stream) != cudaSuccess) return GDA_ERR_CUDA;
        s_end = g_tev[2 * g_tused + 1];
        ++g_tused;
      }
    }
    if (gda::launch_small(ps, small_c, stream) != cudaSuccess) return GDA_ERR_CUDA;
    if (s_end != nullptr && cudaEventRecord(s_end, stream) != cudaSuccess) return GDA_ERR_CUDA;
    return GDA_OK;
  }

  const Layout l = layout(a->B, a->Hq, a->Hkv, a->D, a->num_splits);
  unsigned char* base = static_cast<unsigned char*>(ws);
  const int npass = passes(a->Hq, a->Hkv);
  const bool fp8 = a->kv_dtype == GDA_KV_E4M3;
  const int variant = (a->variant == GDA_VARIANT_SIMT)  ? gda::kVariantSimt
                      : (a->variant == GDA_VARIANT_TMA) ? gda::kVariantTma
                                                        : gda::kVariantMma;
  // G > 8 on the MMA kernel: the groups of 8 query heads in teams of 2 or 3, every
  // group of a team in one piece (one HBM read of the KV head's rows per team); on the
  // FP8 kernel in pairs, except for three groups (a half-empty pair costs a full one, and
  // two pairs measured no faster than three single passes on b64_l4096 lengths: 135.0
  // us for G = 32's two pairs against 135.9 us for G = 24's three passes)
  const int team = (variant != gda::kVariantMma || npass < 2) ? 1 : fp8 ? (npass == 3 ? 1 : 2) : team_size(npass);
  const int nteam = (npass + team - 1) / team;
  // the heads that split the batch into segments for the schedule
  const long long vheads = (long long)a->Hkv * nteam;
  const int min_chunk = a->min_chunk > 0 ? a->min_chunk : kDefaultMinChunk;
  // the rule's e4m3 variant: a position streams in half the time, so the per-CTA bound
  // for the stream schedule is twice as many positions and S_opt comes from 16 S^2 >
  // lmax (half the BF16 count)
  const int kv8 = fp8 ? 1 : 0;
  const int auto_grid = sms < gda::kAutoMaxCtas ? sms : gda::kAutoMaxCtas;
  int splits = a->num_splits > 0 ? a->num_splits : 0;
  if (splits == 0 && a->window == 0 && a->max_len > 0 && a->total_len > 0) {
    // the caller knows a bound on the longest length and the exact total: the rule
    // runs here, and uniform splits launch as explicit ones (no scan of kv_indptr
    // on the device, no idle CTAs)
    splits = host_uniform_splits(a->B, vheads, auto_grid, min_chunk, a->max_len, a->total_len, kv8);
  }
  if (splits == 0 && a->window > 0) {
    // A window bounds every sequence's range by `window`: equal splits of at least
    // min_chunk positions, about one per CTA (this fits the automatic workspace).
    const long long segs = (long long)a->B * vheads;
    const long long by_len = (a->window + min_chunk - 1) / min_chunk;
    const long long by_grid = (auto_grid + segs - 1) / segs;
    splits = (int)(by_len < by_grid ? by_len : by_grid);
    if (splits < 1) splits = 1;
  }
  int grid;
  if (splits > 0) {
    const long long units = (long long)a->B * vheads * splits;
    grid = (int)(units < sms ? units : sms);
  } else {
    grid = auto_grid;
  }

  gda::Stage1Params p1;
  p1.q = reinterpret_cast<const __nv_bfloat16*>(a->q);
  p1.k_pool = reinterpret_cast<const unsigned char*>(a->k_pool);
  p1.v_pool = reinterpret_cast<const unsigned char*>(a->v_pool);
  p1.indptr = a->kv_indptr;
  p1.indices = a->kv_indices;
  p1.o_part = reinterpret_cast<float*>(base + l.o_off);
  p1.lse_part = reinterpret_cast<float*>(base + l.lse_off);
  p1.hdr = reinterpret_cast<gda::WsHeader*>(base);
  p1.num_slots = a->num_slots;
  p1.B = a->B;
  p1.Hq = a->Hq;
  p1.Hkv = a->Hkv;
  p1.G = a->Hq / a->Hkv;
  p1.npass = npass;
  p1.team = team;
  p1.nteam = nteam;
  p1.window = a->window;
  // e4m3 pools: k_descale joins the score scale (one rounding, from double)
  p1.scale_log2 = fp8 ? (float)((double)a->scale * (double)a->k_descale * 1.4426950408889634074)
                      : a->scale * 1.44269504088896340736f;
  p1.v_descale = fp8 ? a->v_descale : 1.0f;
  p1.num_splits = splits;
  p1.min_chunk = min_chunk;
  // automatic stream schedule with more segments than CTAs: a segment start costs a CTA
  // about as much as kPieceCost positions (twice as many positions of an e4m3 cache)
  p1.piece_cost = (splits == 0 && (long long)a->B * vheads > grid) ? (fp8 ? gda::kPieceCostE4m3 : gda::kPieceCost) : 0;
  p1.rule_kv8 = kv8;
  p1.check_indices = a->check_indices ? 1 : 0;
  p1.wait_limit = wait_limit();
  cudaEvent_t t_end = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_tused < g_tmax) {
      if (cudaEventRecord(g_tev[2 * g_tused], stream) != cudaSuccess) return GDA_ERR_CUDA;
      t_end = g_tev[2 * g_tused + 1];
      ++g_tused;
    }
  }
  const cudaError_t le =
      fp8 ? gda::launch_stage1_fp8(p1, grid, stream) : gda::launch_stage1(p1, variant, grid, stream);
  if (le != cudaSuccess) return GDA_ERR_CUDA;
  if (t_end != nullptr && cudaEventRecord(t_end, stream) != cudaSuccess) return GDA_ERR_CUDA;

  gda::Stage2Params p2;
  p2.gate = reinterpret_cast<const __nv_bfloat16*>(a->gate);
  p2.indptr = a->kv_indptr;
  p2.o_part = p1.o_part;
  p2.lse_part = p1.lse_part;
  p2.out = reinterpret_cast<__nv_bfloat16*>(a->out);
  p2.lse_out = a->lse;
  p2.sinks = a->sinks;
  p2.B = a->B;
  p2.Hq = a->Hq;
  p2.Hkv = a->Hkv;
  p2.G = p1.G;
  p2.npass = npass;
  p2.team = team;
  p2.nteam = nteam;
  p2.window = a->window;
  p2.num_splits = p1.num_splits;
  p2.grid1 = grid;
  p2.min_chunk = min_chunk;
  p2.piece_cost = p1.piece_cost;
  p2.rule_kv8 = kv8;
  p2.fuse_gate = a->fuse_gate ? 1 : 0;
  // batched merge: when the B * Hq stage-2 CTAs fit one wave at its register count
  // (six CTAs per SM) and a warp merges more than one partial (automatic splits may)
  p2.batched = ((long long)a->B * a->Hq <= 6LL * sms && (splits == 0 || splits > 4)) ? 1 : 0;
  if (gda::launch_stage2(p2, stream) != cudaSuccess) return GDA_ERR_CUDA;
  return GDA_OK;
}

// Make the internal workspace of the current device at least `need` bytes.  A
// growth allocates a new buffer of at least twice the old size and keeps the old
// one allocated until the process exits, so a graph captured on it stays valid;
// the retired buffers then total less than the current one.
int ensure_workspace(size_t need, cudaStream_t stream, bool check_capture, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ws_bytes >= need) {
    *out = d.ws;
    return GDA_OK;
  }
  if (check_capture) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) return GDA_ERR_CUDA;
    if (st != cudaStreamCaptureStatusNone) return GDA_ERR_CAPTURE;
  }
  const size_t grown = round_up(need > 2 * d.ws_bytes ? need : 2 * d.ws_bytes, 256);
  void* p = nullptr;
  if (cudaMalloc(&p, grown) != cudaSuccess) return GDA_ERR_CUDA;
  // the header (error word) starts at zero before any stream can use the buffer
  if (cudaMemset(p, 0, gda::kHeaderBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(p);
    return GDA_ERR_CUDA;
  }
  if (d.ws) d.retired.push_back(d.ws);
  d.ws = p;
  d.ws_bytes = grown;
  *out = p;
  return GDA_OK;
}

// ---- scratch for gda_decode_noalloc --------------------------------------------
//
// Callers that may not allocate device memory get a fixed scratch area instead of
// the workspace: a file-scope device array, present on every GPU that loads this
// library until the process exits.  In host code g_noalloc_scratch is only a
// stand-in for the symbol; its device address comes from cudaGetSymbolAddress,
// taken once per device with that device current.
__device__ __align__(256) unsigned char g_noalloc_scratch[GDA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device; the first call on a device
// looks it up and clears the header (error word) on `stream`.
int noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return GDA_ERR_CUDA;
    if (cudaMemsetAsync(ptr, 0, gda::kHeaderBytes, stream) != cudaSuccess) return GDA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return GDA_OK;
}

// ---- the library's prefill error word (gda_prefill with error_word == NULL) ---------
__device__ unsigned int g_prefill_error;
unsigned int* g_prefill_error_ptr[kMaxDevices] = {};

int prefill_error_word(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_prefill_error_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    // a zero-initialised __device__ word: nothing to enqueue (so a call refused later,
    // e.g. under capture, leaves no work behind)
    if (cudaGetSymbolAddress(&ptr, g_prefill_error) != cudaSuccess || ptr == nullptr) return GDA_ERR_CUDA;
    g_prefill_error_ptr[dev] = static_cast<unsigned int*>(ptr);
  }
  *out = g_prefill_error_ptr[dev];
  return GDA_OK;
}

}  // namespace

extern "C" {

size_t gda_workspace_bytes(int B, int Hq, int Hkv, int D, int num_splits) {
  if (check_sizes(B, Hq, Hkv, D, num_splits) != GDA_OK) return 0;
  return layout(B, Hq, Hkv, D, num_splits).total;
}

int gda_workspace_init(void* workspace, size_t workspace_bytes, gda_stream_t stream) {
  if (workspace == nullptr) return GDA_ERR_NULL;
  if (!aligned(workspace, 256)) return GDA_ERR_ALIGN;
  if (workspace_bytes < (size_t)gda::kHeaderBytes) return GDA_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, gda::kHeaderBytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDA_ERR_CUDA;
  return GDA_OK;
}

int gda_decode_ex(const gda_args* args, void* workspace, size_t workspace_bytes, gda_stream_t stream) {
  int rc = validate_args(args);
  if (rc != GDA_OK) return rc;
  if (args->B == 0) return GDA_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return GDA_ERR_WORKSPACE;
  if (workspace_bytes < gda_workspace_bytes(args->B, args->Hq, args->Hkv, args->D, args->num_splits))
    return GDA_ERR_WORKSPACE;
  return enqueue(args, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int gda_decode(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k_pool, const gda_bf16* v_pool,
               const int32_t* kv_indptr, const int32_t* kv_indices, gda_bf16* out, int B, int Hq, int Hkv, int D,
               float scale, int num_splits, gda_stream_t stream) {
  gda_args a = {};
  a.q = q;
  a.gate = gate;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.out = out;
  a.lse = nullptr;
  a.num_slots = 0;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.num_splits = num_splits;
  a.fuse_gate = 1;
  a.check_indices = 0;
  a.variant = GDA_VARIANT_AUTO;
  a.min_chunk = 0;
  a.window = 0;
  a.sinks = nullptr;
  int rc = validate_args(&a);
  if (rc != GDA_OK) return rc;
  if (B == 0) return GDA_OK;
  void* ws = nullptr;
  const size_t need = gda_workspace_bytes(B, Hq, Hkv, D, num_splits);
  rc = ensure_workspace(need, reinterpret_cast<cudaStream_t>(stream), true, &ws);
  if (rc != GDA_OK) return rc;
  return enqueue(&a, ws, reinterpret_cast<cudaStream_t>(stream));
}

int gda_decode_e4m3(const gda_bf16* q, const gda_bf16* gate, const uint8_t* k_pool, const uint8_t* v_pool,
                    const int32_t* kv_indptr, const int32_t* kv_indices, gda_bf16* out, int B, int Hq, int Hkv,
                    int D, float scale, float k_descale, float v_descale, int num_splits, gda_stream_t stream) {
  gda_args a = {};
  a.q = q;
  a.gate = gate;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.out = out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.num_splits = num_splits;
  a.fuse_gate = 1;
  a.variant = GDA_VARIANT_AUTO;
  a.kv_dtype = GDA_KV_E4M3;
  a.k_descale = k_descale;
  a.v_descale = v_descale;
  int rc = validate_args(&a);
  if (rc != GDA_OK) return rc;
  if (B == 0) return GDA_OK;
  void* ws = nullptr;
  const size_t need = gda_workspace_bytes(B, Hq, Hkv, D, num_splits);
  rc = ensure_workspace(need, reinterpret_cast<cudaStream_t>(stream), true, &ws);
  if (rc != GDA_OK) return rc;
  return enqueue(&a, ws, reinterpret_cast<cudaStream_t>(stream));
}

int gda_decode_noalloc(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k_pool, const gda_bf16* v_pool,
                       const int32_t* kv_indptr, const int32_t* kv_indices, gda_bf16* out, int B, int Hq, int Hkv,
                       int D, float scale, int num_splits, gda_stream_t stream) {
  gda_args a = {};
  a.q = q;
  a.gate = gate;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = kv_indptr;
  a.kv_indices = kv_indices;
  a.out = out;
  a.lse = nullptr;
  a.num_slots = 0;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.num_splits = num_splits;
  a.fuse_gate = 1;
  a.check_indices = 0;
  a.variant = GDA_VARIANT_AUTO;
  a.min_chunk = 0;
  a.window = 0;
  a.sinks = nullptr;
  int rc = validate_args(&a);
  if (rc != GDA_OK) return rc;
  if (B == 0) return GDA_OK;
  if (gda_workspace_bytes(B, Hq, Hkv, D, num_splits) > (size_t)GDA_NOALLOC_SCRATCH_BYTES) return GDA_ERR_WORKSPACE;
  void* ws = nullptr;
  rc = noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &ws);
  if (rc != GDA_OK) return rc;
  return enqueue(&a, ws, reinterpret_cast<cudaStream_t>(stream));
}

int gda_qk_norm_rope_kv_write(const gda_bf16* qgkv, int64_t row_stride, const gda_bf16* w_q_norm,
                              const gda_bf16* w_k_norm, float eps, const gda_bf16* cos_t, const gda_bf16* sin_t,
                              int rope_dim, const int32_t* slots, int64_t num_slots, gda_bf16* q_out,
                              gda_bf16* gate_out, gda_bf16* k_pool, gda_bf16* v_pool, int B, int Hq, int Hkv, int D,
                              gda_stream_t stream) {
  if (B < 0 || Hq < 1 || Hkv < 1 || D < 1 || num_slots < 0) return GDA_ERR_SHAPE;
  if (row_stride < (int64_t)(2 * Hq + 2 * Hkv) * D) return GDA_ERR_SHAPE;
  if (rope_dim < 0 || rope_dim > D) return GDA_ERR_SHAPE;
  if (D != gda::kD || rope_dim % 16 != 0) return GDA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f)) return GDA_ERR_SHAPE;
  if (B == 0) return GDA_OK;
  if (!qgkv || !slots || !q_out || !k_pool || !v_pool) return GDA_ERR_NULL;
  if (rope_dim > 0 && (!cos_t || !sin_t)) return GDA_ERR_NULL;
  if (!aligned(qgkv, 16) || row_stride % 8 != 0 || !aligned(q_out, 16) || !aligned(k_pool, 16) ||
      !aligned(v_pool, 16) || (gate_out && !aligned(gate_out, 16)) || (w_q_norm && !aligned(w_q_norm, 16)) ||
      (w_k_norm && !aligned(w_k_norm, 16)) || (cos_t && !aligned(cos_t, 16)) || (sin_t && !aligned(sin_t, 16)) ||
      !aligned(slots, 4))
    return GDA_ERR_ALIGN;
  gda::PrepParams p;
  p.qgkv = reinterpret_cast<const __nv_bfloat16*>(qgkv);
  p.row_stride = row_stride;
  p.w_q = reinterpret_cast<const __nv_bfloat16*>(w_q_norm);
  p.w_k = reinterpret_cast<const __nv_bfloat16*>(w_k_norm);
  p.eps = eps;
  p.cos_t = reinterpret_cast<const __nv_bfloat16*>(cos_t);
  p.sin_t = reinterpret_cast<const __nv_bfloat16*>(sin_t);
  p.rope_dim = rope_dim;
  p.slots = slots;
  p.num_slots = num_slots;
  p.q_out = reinterpret_cast<__nv_bfloat16*>(q_out);
  p.gate_out = reinterpret_cast<__nv_bfloat16*>(gate_out);
  p.k_pool = reinterpret_cast<__nv_bfloat16*>(k_pool);
  p.v_pool = reinterpret_cast<__nv_bfloat16*>(v_pool);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  if (gda::launch_prep(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GDA_ERR_CUDA;
  return GDA_OK;
}

int gda_prefill(const gda_bf16* q, const gda_bf16* gate, const gda_bf16* k, const gda_bf16* v,
                const int32_t* kv_lens, gda_bf16* out, float* lse, int B, int Sq, int Skv, int Hq, int Hkv,
                int D, float scale, int causal, uint32_t* error_word, gda_stream_t stream) {
  if (B < 0 || Sq < 0 || Skv < 0 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return GDA_ERR_SHAPE;
  if (D != gda::kD) return GDA_ERR_UNSUPPORTED;
  if (!isfinite(scale) || !(scale > 0.0f)) return GDA_ERR_ARG;
  if (B == 0 || Sq == 0) return GDA_OK;
  if (!q || !out || (Skv > 0 && (!k || !v))) return GDA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(out, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
      (gate && !aligned(gate, 16)) || (kv_lens && !aligned(kv_lens, 4)) || (lse && !aligned(lse, 4)) ||
      (error_word && !aligned(error_word, 4)))
    return GDA_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* err = error_word;
  if (err == nullptr) {
    int rc = prefill_error_word(&err);
    if (rc != GDA_OK) return rc;
  }
  gda::PrefillParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
  p.kv_lens = kv_lens;
  p.error = err;
  p.B = B;
  p.Sq = Sq;
  p.Skv = Skv;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.scale_log2 = scale * 1.44269504088896340736f;
  p.causal = causal ? 1 : 0;
  p.fuse_gate = gate ? 1 : 0;
  p.wait_limit = wait_limit();
  // with Skv == 0 the key maps still need a valid base: the queries' (never loaded)
  const void* kb = Skv > 0 ? static_cast<const void*>(k) : static_cast<const void*>(q);
  const void* vb = Skv > 0 ? static_cast<const void*>(v) : static_cast<const void*>(q);
  const cudaError_t le = gda::launch_prefill(p, q, kb, vb, gate, s);
  if (le == cudaErrorStreamCaptureUnsupported) return GDA_ERR_CAPTURE;  // first use while capturing
  if (le != cudaSuccess) return GDA_ERR_CUDA;
  return GDA_OK;
}

int gda_prefill_read_error(gda_stream_t stream, int clear, uint32_t* error_word) {
  if (error_word == nullptr) return GDA_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* dev_word = nullptr;
  int rc = prefill_error_word(&dev_word);
  if (rc != GDA_OK) return rc;
  unsigned int w = 0;
  if (cudaMemcpyAsync(&w, dev_word, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDA_ERR_CUDA;
  if (clear && w != 0) {
    if (cudaMemsetAsync(dev_word, 0, sizeof(w), s) != cudaSuccess) return GDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDA_ERR_CUDA;
  }
  *error_word = w;
  return w == 0 ? GDA_OK : GDA_ERR_DEVICE;
}

int gda_reserve(int max_B, int Hq, int Hkv, int D, int max_splits) {
  int rc = check_sizes(max_B, Hq, Hkv, D, max_splits);
  if (rc != GDA_OK) return rc;
  // the automatic mode and every explicit split count up to max_splits must fit
  size_t need = gda_workspace_bytes(max_B, Hq, Hkv, D, 0);
  if (max_splits > 0) {
    const size_t e = gda_workspace_bytes(max_B, Hq, Hkv, D, max_splits);
    if (e > need) need = e;
  }
  void* ws = nullptr;
  return ensure_workspace(need, nullptr, false, &ws);
}

int gda_auto_splits(int B, int heads, int grid, int min_chunk, int lmax, int64_t total) {
  if (B < 0 || heads < 1 || grid < 1 || lmax < 0 || total < 0) return -1;
  return host_uniform_splits(B, heads, grid, min_chunk > 0 ? min_chunk : kDefaultMinChunk, lmax, total, 0);
}

int gda_small_path_cluster(int64_t pairs, int max_len) {
  if (pairs < 0) return 0;
  return gda::small_cluster_for((long long)pairs, max_len);
}

size_t gda_step_layout(int B, int Hq, int D, int64_t nnz, size_t offsets[4]) {
  if (offsets == nullptr || B < 1 || Hq < 1 || D < 1 || nnz < 0) return 0;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t qg = (size_t)B * Hq * D * sizeof(gda_bf16);
  offsets[0] = 0;
  offsets[1] = up(qg);
  offsets[2] = offsets[1] + up(qg);
  offsets[3] = offsets[2] + up((size_t)(B + 1) * sizeof(int32_t));
  return offsets[3] + up((size_t)nnz * sizeof(int32_t));
}

int gda_decode_step_host(const void* host_in, void* dev_in, size_t in_bytes, const void* k_pool,
                         const void* v_pool, int kv_dtype, float k_descale, float v_descale, gda_bf16* dev_out,
                         void* host_out, int B, int Hq, int Hkv, int D, int64_t nnz, float scale, int num_splits,
                         int flags, int synchronize, gda_stream_t stream) {
  if (B < 0 || nnz < 0) return GDA_ERR_SHAPE;
  if ((flags & ~(GDA_STEP_MAP_IN | GDA_STEP_MAP_OUT)) != 0) return GDA_ERR_ARG;
  if (B == 0) return GDA_OK;
  size_t off[4];
  const size_t total = gda_step_layout(B, Hq, D, nnz, off);
  if (total == 0) return GDA_ERR_SHAPE;
  if (in_bytes != total) return GDA_ERR_SHAPE;
  const bool map_in = (flags & GDA_STEP_MAP_IN) != 0, map_out = (flags & GDA_STEP_MAP_OUT) != 0;
  if (host_in == nullptr || host_out == nullptr || (!map_in && dev_in == nullptr) || (!map_out && dev_out == nullptr))
    return GDA_ERR_NULL;
  if (!aligned(host_in, 256) && map_in) return GDA_ERR_ALIGN;
  if (!map_in && !aligned(dev_in, 256)) return GDA_ERR_ALIGN;
  // the decode's own checks on the views, with placeholder bases for mapped memory
  // (whose device addresses are only known after a CUDA query), so a bad call
  // enqueues nothing
  const unsigned char* din = static_cast<const unsigned char*>(map_in ? host_in : dev_in);
  gda_args a = {};
  a.q = reinterpret_cast<const gda_bf16*>(din + off[0]);
  a.gate = reinterpret_cast<const gda_bf16*>(din + off[1]);
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.kv_indptr = reinterpret_cast<const int32_t*>(din + off[2]);
  a.kv_indices = reinterpret_cast<const int32_t*>(din + off[3]);
  a.out = map_out ? static_cast<gda_bf16*>(host_out) : dev_out;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.scale = scale;
  a.num_splits = num_splits;
  a.fuse_gate = 1;
  a.variant = GDA_VARIANT_AUTO;
  a.kv_dtype = kv_dtype;
  a.k_descale = k_descale;
  a.v_descale = v_descale;
  a.total_len = nnz;  // kv_indptr[B] == nnz; max_len is read below
  int rc = validate_args(&a);
  if (rc != GDA_OK) return rc;
  // kv_indptr is in host memory here (B + 1 values): check it before anything is
  // enqueued, since the kernels would otherwise read kv_indices past the end of the
  // block, and take the longest length as the dispatch's exact bound
  {
    const int32_t* hp = reinterpret_cast<const int32_t*>(static_cast<const unsigned char*>(host_in) + off[2]);
    if (hp[0] != 0 || (int64_t)hp[B] != nnz) return GDA_ERR_SHAPE;
    long long lmax = 0;
    for (int b = 0; b < B; ++b) {
      const long long d = (long long)hp[b + 1] - (long long)hp[b];
      if (d < 0) return GDA_ERR_SHAPE;
      if (d > lmax) lmax = d;
    }
    a.max_len = (int)(lmax < 0x7FFFFFFF ? lmax : 0x7FFFFFFF);
  }
  // mapped host memory: the device address of each pointer (page-locked host memory only)
  auto device_view = [](const void* h, void** d) -> int {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, h) != cudaSuccess) {
      (void)cudaGetLastError();
      return GDA_ERR_ARG;
    }
    if (pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr) return GDA_ERR_ARG;
    *d = pa.devicePointer;
    return GDA_OK;
  };
  if (map_in) {
    void* d = nullptr;
    rc = device_view(host_in, &d);
    if (rc != GDA_OK) return rc;
    const unsigned char* db = static_cast<const unsigned char*>(d);
    a.q = reinterpret_cast<const gda_bf16*>(db + off[0]);
    a.gate = reinterpret_cast<const gda_bf16*>(db + off[1]);
    a.kv_indptr = reinterpret_cast<const int32_t*>(db + off[2]);
    a.kv_indices = reinterpret_cast<const int32_t*>(db + off[3]);
  }
  if (map_out) {
    void* d = nullptr;
    rc = device_view(host_out, &d);
    if (rc != GDA_OK) return rc;
    if (!aligned(d, 16)) return GDA_ERR_ALIGN;
    a.out = static_cast<gda_bf16*>(d);
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  rc = ensure_workspace(gda_workspace_bytes(B, Hq, Hkv, D, num_splits), st, true, &ws);
  if (rc != GDA_OK) return rc;
  if (!map_in && cudaMemcpyAsync(dev_in, host_in, total, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return GDA_ERR_CUDA;
  rc = enqueue(&a, ws, st);
  if (rc != GDA_OK) return rc;
  const size_t out_bytes = (size_t)B * Hq * D * sizeof(gda_bf16);
  if (!map_out && cudaMemcpyAsync(host_out, dev_out, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return GDA_ERR_CUDA;
  if (synchronize && cudaStreamSynchronize(st) != cudaSuccess) return GDA_ERR_CUDA;
  return GDA_OK;
}

int gda_gate(const gda_bf16* o, const gda_bf16* gate, gda_bf16* out, int64_t n, gda_stream_t stream) {
  if (n < 0) return GDA_ERR_SHAPE;
  if (n == 0) return GDA_OK;
  if (!o || !gate || !out) return GDA_ERR_NULL;
  if (!aligned(o, 16) || !aligned(gate, 16) || !aligned(out, 16)) return GDA_ERR_ALIGN;
  if (gda::launch_gate(reinterpret_cast<const __nv_bfloat16*>(o), reinterpret_cast<const __nv_bfloat16*>(gate),
                       reinterpret_cast<__nv_bfloat16*>(out), (long long)n,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDA_ERR_CUDA;
  return GDA_OK;
}

int gda_read_error(const void* workspace, gda_stream_t stream, int clear, uint32_t* error_word) {
  if (error_word == nullptr) return GDA_ERR_NULL;
  const void* ws = workspace;
  if (ws == nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    ws = g_dev[dev].ws;
  }
  if (ws == nullptr) {
    *error_word = 0;
    return GDA_OK;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int w = 0;
  if (cudaMemcpyAsync(&w, ws, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDA_ERR_CUDA;
  if (clear && w != 0) {
    if (cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(w), s) != cudaSuccess) return GDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDA_ERR_CUDA;
  }
  *error_word = w;
  return w == 0 ? GDA_OK : GDA_ERR_DEVICE;
}

int gda_timing_begin(int max_calls) {
  if (max_calls < 0) return GDA_ERR_SHAPE;
  std::lock_guard<std::mutex> lk(g_mu);
  for (cudaEvent_t e : g_tev) cudaEventDestroy(e);
  g_tev.clear();
  g_tmax = g_tused = 0;
  g_tev.resize(2 * (size_t)max_calls, nullptr);
  for (size_t i = 0; i < g_tev.size(); ++i) {
    if (cudaEventCreate(&g_tev[i]) != cudaSuccess) {
      for (size_t j = 0; j < i; ++j) cudaEventDestroy(g_tev[j]);
      g_tev.clear();
      return GDA_ERR_CUDA;
    }
  }
  g_tmax = max_calls;
  return GDA_OK;
}

int gda_timing_end(int* n_timed, double* total_ms) {
  if (n_timed == nullptr || total_ms == nullptr) return GDA_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_mu);
  double sum = 0.0;
  int rc = GDA_OK;
  for (int i = 0; i < g_tused; ++i) {
    float ms = 0.0f;
    if (cudaEventSynchronize(g_tev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_tev[2 * i], g_tev[2 * i + 1]) != cudaSuccess) {
      rc = GDA_ERR_CUDA;
      break;
    }
    sum += ms;
  }
  *n_timed = rc == GDA_OK ? g_tused : 0;
  *total_ms = rc == GDA_OK ? sum : 0.0;
  for (cudaEvent_t e : g_tev) cudaEventDestroy(e);
  g_tev.clear();
  g_tmax = g_tused = 0;
  return rc;
}

const char* gda_status_str(int status) {
  switch (status) {
    case GDA_OK: return "GDA_OK: success";
    case GDA_ERR_NULL: return "GDA_ERR_NULL: a required pointer is NULL";
    case GDA_ERR_ALIGN: return "GDA_ERR_ALIGN: a pointer is not aligned (16 bytes for bf16 tensors, 4 for indices)";
    case GDA_ERR_SHAPE: return "GDA_ERR_SHAPE: invalid sizes (B<0, Hq<1, Hkv<1, Hq%Hkv!=0, negative count)";
    case GDA_ERR_UNSUPPORTED: return "GDA_ERR_UNSUPPORTED: shape or option not served by the built kernels (D = 256)";
    case GDA_ERR_SPLITS: return "GDA_ERR_SPLITS: num_splits exceeds GDA_MAX_SPLITS";
    case GDA_ERR_WORKSPACE: return "GDA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case GDA_ERR_CAPTURE: return "GDA_ERR_CAPTURE: workspace growth requested while the stream is capturing";
    case GDA_ERR_CUDA: return "GDA_ERR_CUDA: a CUDA call or kernel launch failed";
    case GDA_ERR_DEVICE: return "GDA_ERR_DEVICE: a kernel flagged an error in the workspace error word";
    case GDA_ERR_ARG: return "GDA_ERR_ARG: a scalar argument is outside its domain (non-finite descale)";
    default: return "unknown gda status";
  }
}

int gda_debug_wait_limit(int64_t cycles) {
  g_wait_limit.store(cycles > 0 && cycles < gda::kWaitLimitCycles ? (long long)cycles : 0);
  return GDA_OK;
}

int gda_version(void) { return 300; }  // 0.3.0: gda_debug_wait_limit

}  // extern "C"
