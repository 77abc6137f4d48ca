// api.cu -- the C ABI of libtg.so (include/tg.h): argument checks, the
// per-device context (SM count, status word, wait limit), the shape-keyed
// tile table and the dispatch of every product onto its kernels.
#include <cuda_runtime.h>
#include <dlfcn.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <fstream>
#include <mutex>
#include <shared_mutex>
#include <sstream>
#include <string>
#include <unordered_map>

#include "attn.h"
#include "ptx.cuh"
#include "tg.h"
#include "tg_internal.h"

namespace tg {

// ------------------------------------------------------------ status word
// One word per device (a module global exists once per device context).
// Kernels OR a code into it when a bounded wait runs out.
__device__ unsigned int g_status_word;

__global__ void wait_probe_kernel(unsigned long long timeout_ns, unsigned int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: this wait can only end by timing out
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, timeout_ns, &abort_flag, status, 0x7e);
  __syncthreads();
}

cudaError_t wait_probe_launch(unsigned long long timeout_ns, unsigned int* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("TG_PDL");
    return !(e && strcmp(e, "0") == 0);
  }();
  return on;
}

bool chunked_mn_enabled() {
  static const bool on = [] {
    const char* e = getenv("TG_CHUNKED_MN");
    return !(e && strcmp(e, "0") == 0);
  }();
  return on;
}

// FP32 operands on the tensor cores (three-part split) when the pitches allow
// (default), or always on the CUDA cores ($TG_FP32_PATH=ffma).
static bool fp32_tc_enabled() {
  static const bool on = [] {
    const char* e = getenv("TG_FP32_PATH");
    return !(e && strcmp(e, "ffma") == 0);
  }();
  return on;
}

struct DevCtx {
  bool ready = false;
  tg_status init_status = TG_OK;
  int sms = 0;
  unsigned int* status = nullptr;
  unsigned long long timeout_ns = 2000000000ull;
};

static std::mutex g_ctx_mu;
static DevCtx g_ctx[128];

static tg_status device_ctx(DevCtx** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return TG_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  DevCtx& c = g_ctx[dev];
  if (!c.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TG_ERR_CUDA;
    if (major != 10 || minor != 3) {
      c.init_status = TG_ERR_UNSUPPORTED_DEVICE;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return TG_ERR_CUDA;
      c.status = static_cast<unsigned int*>(p);
      if (const char* e = getenv("TG_WAIT_TIMEOUT_MS")) {
        long v = strtol(e, nullptr, 10);
        if (v > 0 && v < 600000) c.timeout_ns = static_cast<unsigned long long>(v) * 1000000ull;
      }
    }
    c.ready = true;
  }
  *out = &c;
  return c.init_status;
}

// ------------------------------------------------------------- call record
static thread_local std::string t_last_call;
static int log_enabled() {
  static int v = [] {
    const char* e = getenv("TG_LOG");
    return (e && *e && strcmp(e, "0") != 0) ? 1 : 0;
  }();
  return v;
}
static void record(const std::string& s) {
  t_last_call = s;
  if (log_enabled()) fprintf(stderr, "[tg] %s\n", s.c_str());
}
void note_last_call(const std::string& s) { record(s); }

// -------------------------------------------------------------- tile table
struct TableKey {
  int layout, in, out;
  int64_t M, N, K, batch;
  bool operator==(const TableKey& o) const {
    return layout == o.layout && in == o.in && out == o.out && M == o.M && N == o.N && K == o.K &&
           batch == o.batch;
  }
};
struct TableKeyHash {
  size_t operator()(const TableKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const int64_t v[7] = {k.layout, k.in, k.out, k.M, k.N, k.K, k.batch};
    for (int64_t x : v) h = (h ^ static_cast<uint64_t>(x)) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
struct TableVal {
  int bn, splits, raster;  // splits 0 = stream-K; raster: -1 = by operand size, 0 = along M, 1 = along N
  int tail;                // > 1: tail split of the tiles past the last whole wave
  int pair;                // 1: CTA-pair kernel (256-row tiles)
  int csplit;              // > 1: split-K across the CTAs of a cluster
};
static std::shared_mutex g_table_mu;
static std::unordered_map<TableKey, TableVal, TableKeyHash> g_table;
static std::once_flag g_table_env_once;

static const char* layout_name(int l) { return l == LAYOUT_NT ? "nt" : (l == LAYOUT_NN ? "nn" : "tn"); }
static int parse_layout(const std::string& s) {
  if (s == "nt" || s == "fwd") return LAYOUT_NT;
  if (s == "nn" || s == "dgrad") return LAYOUT_NN;
  if (s == "tn" || s == "wgrad") return LAYOUT_TN;
  return -1;
}
static int parse_dtype(const std::string& s) {
  if (s == "bf16") return TG_BF16;
  if (s == "f16" || s == "fp16") return TG_F16;
  if (s == "f32" || s == "fp32") return TG_F32;
  return -1;
}

static tg_status load_table_file(const char* path) {
  std::unordered_map<TableKey, TableVal, TableKeyHash> t;
  if (path && *path) {
    std::ifstream f(path);
    if (!f) return TG_ERR_TABLE;
    std::string line;
    while (std::getline(f, line)) {
      const size_t h = line.find('#');
      if (h != std::string::npos) line.resize(h);
      std::istringstream ss(line);
      std::string op, din, dout, bs, sp;
      int64_t M, N, K, batch;
      int bn, splits, tail = 0, pair = 0, csplit = 0;
      if (!(ss >> op)) continue;  // blank line
      if (!(ss >> din >> dout >> M >> N >> K >> batch >> bs >> sp)) return TG_ERR_TABLE;
      {  // tile width, "p" suffix: CTA pair (256 x bn tiles)
        char* endp = nullptr;
        const long v = strtol(bs.c_str(), &endp, 10);
        if (endp == bs.c_str()) return TG_ERR_TABLE;
        if (*endp == 'p' && endp[1] == '\0') pair = 1;
        else if (*endp != '\0') return TG_ERR_TABLE;
        bn = static_cast<int>(v);
      }
      if (sp == "sk") {
        splits = 0;
      } else if (sp.size() > 1 && sp[0] == 'c') {  // cluster split-K: cN
        char* endp = nullptr;
        const long v = strtol(sp.c_str() + 1, &endp, 10);
        if (*endp != '\0' || v < 2 || v > 8) return TG_ERR_TABLE;
        splits = 1;
        csplit = static_cast<int>(v);
      } else if (sp.size() > 1 && sp[0] == 't') {  // tail split: tN
        char* endp = nullptr;
        const long v = strtol(sp.c_str() + 1, &endp, 10);
        if (*endp != '\0' || v < 2 || v > 64) return TG_ERR_TABLE;
        splits = 1;
        tail = static_cast<int>(v);
      } else {
        char* endp = nullptr;
        const long v = strtol(sp.c_str(), &endp, 10);
        if (endp == sp.c_str() || *endp != '\0') return TG_ERR_TABLE;
        splits = static_cast<int>(v);
      }
      std::string rs;
      int raster = -1;
      if (ss >> rs) {
        if (rs == "m") raster = 0;
        else if (rs == "n") raster = 1;
        else if (rs != "auto") return TG_ERR_TABLE;
      }
      const int l = parse_layout(op), i = parse_dtype(din), o = parse_dtype(dout);
      if (l < 0 || i < 0 || o < 0 || M <= 0 || N <= 0 || K <= 0 || batch <= 0) return TG_ERR_TABLE;
      if (!(bn == 64 || bn == 128 || bn == 144 || bn == 192 || bn == 256) || splits < 0 || splits > 64)
        return TG_ERR_TABLE;
      if (bn % 64 != 0 && (splits == 0 || tail > 0)) return TG_ERR_TABLE;  // partial tiles: 64-column multiples
      if (pair && (bn == 64 || bn == 144)) return TG_ERR_TABLE;  // pairs: widths 128, 192, 256
      if (csplit && (pair || bn == 144)) return TG_ERR_TABLE;    // cluster split: single CTAs, 64..256
      t[TableKey{l, i, o, M, N, K, batch}] = TableVal{bn, splits, raster, tail, pair, csplit};
    }
  }
  std::unique_lock<std::shared_mutex> lk(g_table_mu);
  g_table.swap(t);
  return TG_OK;
}

// At first use: $TG_TABLE if set (empty = no table), else the table shipped
// next to the library (tables/gb300.txt beside libtg.so), if present.
static void table_env_init() {
  std::call_once(g_table_env_once, [] {
    if (const char* p = getenv("TG_TABLE")) {
      load_table_file(p);
      return;
    }
    Dl_info info;
    if (dladdr(reinterpret_cast<void*>(&table_env_init), &info) && info.dli_fname) {
      std::string path(info.dli_fname);
      const size_t slash = path.rfind('/');
      path = (slash == std::string::npos ? std::string(".") : path.substr(0, slash)) + "/tables/gb300.txt";
      std::ifstream f(path);
      if (f.good()) load_table_file(path.c_str());
    }
  });
}

static bool table_lookup(const TableKey& k, TableVal* v) {
  table_env_init();
  std::shared_lock<std::shared_mutex> lk(g_table_mu);
  auto it = g_table.find(k);
  if (it == g_table.end()) return false;
  *v = it->second;
  return true;
}

// ----------------------------------------------------------------- planning
struct Plan {
  int bn = 256;
  int splits = 1;
  int raster_n = 0;
  bool sk = false;  // stream-K schedule (splits is then 1)
  int tail = 0;     // > 1: tail split (splits is then 1)
  bool pair = false;  // CTA-pair kernel: 256 x bn tiles
  int csplit = 0;     // > 1: split-K across a cluster of this many CTAs (splits is then 1)
  bool from_table = false;
};

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Cost model of the persistent tensor-core kernel used when the table has no
// entry: waves of units x (K blocks per unit x block time, or the epilogue
// time when that is longer) + the reduction of split partials.
static Plan heuristic_plan(int64_t M, int64_t N, int64_t K, int64_t batch, int out_bytes, int sms) {
  Plan best;
  double best_t = 1e300;
  const int64_t kb = cdiv(K, 64);
  // narrow first: a wider tile must beat a narrower one by a margin (equal
  // costs mean the same number of tiles, and then the wider one only wastes
  // columns)
  const int bns[5] = {64, 128, 144, 192, 256};
  // one 128 x bn x 64 block: four 128 x bn x 16 MMAs, measured at >= 88 cycles
  // each and ~0.525 * bn cycles from bn = 192 up (the tensor pipe's full
  // rate), or the time the SM's operand feed takes for the block's bytes
  // (16 KB of A and bn rows of B, whole 64-column chunks), ~75 bytes per
  // cycle as measured on the single-CTA kernel: ~600 cycles per block at
  // widths 144 to 256 alike
  auto kb_cycles = [](int bn) {
    const double feed = (16384.0 + 128.0 * 64 * ((bn + 63) / 64)) / 75.0;
    return fmax(4.0 * fmax(88.0, 0.525 * bn), feed);
  };
  for (int bn : bns) {
    const int64_t tiles = batch * cdiv(M, 128) * cdiv(N, bn);
    const double kb_cyc = kb_cycles(bn);
    const double epi_cyc = 128.0 * bn * out_bytes / 48.0;
    for (int64_t s = 1; s <= 32 && s <= kb; ++s) {
      const int64_t kps = cdiv(kb, s);
      const int64_t real = cdiv(kb, kps);
      if (real != s) continue;
      const int64_t units = tiles * s;
      const int64_t waves = cdiv(units, sms);
      double t = waves * (fmax(kps * kb_cyc, s > 1 ? 128.0 * bn * 4 / 48.0 : epi_cyc) + 600.0);
      // the ordered reduction: a second launch plus its pass over the partials
      if (s > 1) t += 5000.0 + (s + 1.0) * M * N * batch * 4.0 / (sms * 24.0);
      if (t < best_t * 0.98) {
        best_t = t;
        best.bn = bn;
        best.splits = static_cast<int>(s);
      }
    }
  }
  // tail split: whole tiles in full waves, the last partial wave's tiles cut along K
  for (int bn : bns) {
    if (bn % 64 != 0) continue;
    const int64_t tiles = batch * cdiv(M, 128) * cdiv(N, bn);
    if (tiles <= sms || tiles % sms == 0) continue;
    const int64_t rem = tiles % sms;
    const double kb_cyc = kb_cycles(bn);
    for (int ts : {2, 3, 4, 6, 8}) {
      const int64_t kps = cdiv(kb, ts), real = cdiv(kb, kps);
      if (real < 2) continue;
      double t = (tiles / sms) * (kb * kb_cyc + 600.0) + cdiv(rem * real, sms) * (kps * kb_cyc + 128.0 * bn * 4 / 48.0 + 600.0);
      t += 8000.0 + rem * real * 128.0 * bn * 4 / (sms * 24.0);  // + the reduce launch
      if (t < best_t * 0.97) {
        best_t = t;
        best.bn = bn;
        best.splits = 1;
        best.sk = false;
        best.tail = static_cast<int>(ts);
      }
    }
  }
  // split-K across a cluster (one wave: tiles x S CTAs at most one per SM,
  // and no more clusters than fit at once: a cluster lives inside one GPC,
  // so on 152 SMs only about 74 / 46 / 36 / 28 / 24 / 20 / 16 clusters of
  // 2..8 are resident together, measured for 3 and 4); the S partial tiles
  // are added through distributed shared memory at ~16 bytes per cycle per
  // SM, after two cluster barriers and the accumulator copy
  for (int bn : {64, 128, 192, 256}) {
    const int64_t tiles = batch * cdiv(M, 128) * cdiv(N, bn);
    const double kb_cyc = kb_cycles(bn);
    for (int64_t cs = 2; cs <= 8 && cs <= kb; ++cs) {
      static const int fit152[9] = {0, 0, 74, 46, 36, 28, 24, 20, 16};
      const int64_t kps = cdiv(kb, cs);
      if (cdiv(kb, kps) != cs || tiles * cs > sms || tiles > fit152[cs] * sms / 152) continue;
      const double t = kps * kb_cyc + 600.0 + 3000.0 + 128.0 * bn * 4 * (cs - 1) / (cs * 16.0);
      if (t < best_t * 0.95) {
        best_t = t;
        best.bn = bn;
        best.splits = 1;
        best.sk = false;
        best.tail = 0;
        best.pair = false;
        best.csplit = static_cast<int>(cs);
      }
    }
  }
  // CTA pairs with the tail split: whole 256 x 256 tiles in full waves of
  // sms / 2 pairs (in lockstep over K), the last partial wave's tiles cut
  // along K into pieces added by the ordered reduction
  if (M > 128) {
    const int bn = 256, pairs = sms / 2;
    const int64_t tiles = batch * cdiv(M, 256) * cdiv(N, bn);
    const double kb_cyc = 4.0 * 0.525 * bn;
    if (pairs > 0 && tiles > pairs && tiles % pairs) {
      const int64_t rem = tiles % pairs;
      for (int ts : {2, 4, 8, 13}) {
        const int64_t kps = cdiv(kb, ts), real = cdiv(kb, kps);
        if (real < 2) continue;
        double t = (tiles / pairs) * (kb * kb_cyc + 600.0) +
                   cdiv(rem * real, pairs) * (kps * kb_cyc + 128.0 * bn * 4 / 48.0 + 600.0);
        t += 8000.0 + rem * real * 256.0 * bn * 4 / (sms * 24.0);
        if (t < best_t * 0.97) {
          best_t = t;
          best.bn = bn;
          best.splits = 1;
          best.sk = false;
          best.tail = ts;
          best.pair = true;
          best.csplit = 0;
        }
      }
    }
  }
  // CTA pairs (256 x bn tiles on two SMs, half of B per SM): a pair MMA
  // costs at least ~125 cycles whatever its width, and runs at the full rate
  // at bn = 256, measured
  for (int bn : {256, 192}) {
    if (M <= 128) break;
    const int64_t tiles = batch * cdiv(M, 256) * cdiv(N, bn);
    const double kb_cyc = 4.0 * fmax(125.0, 0.525 * bn);
    const double epi_cyc = 128.0 * bn * out_bytes / 48.0;
    for (int64_t s = 1; s <= 8 && s <= kb; ++s) {
      const int64_t kps = cdiv(kb, s);
      if (cdiv(kb, kps) != s) continue;
      const int64_t waves = cdiv(tiles * s, sms / 2);
      double t = waves * (fmax(kps * kb_cyc, s > 1 ? 128.0 * bn * 4 / 48.0 : epi_cyc) + 600.0);
      if (s > 1) t += 5000.0 + (s + 1.0) * M * N * batch * 4.0 / (sms * 24.0);
      if (t < best_t * 0.98) {
        best_t = t;
        best.bn = bn;
        best.splits = static_cast<int>(s);
        best.sk = false;
        best.tail = 0;
        best.pair = true;
        best.csplit = 0;
      }
    }
  }
  // Stream-K is never proposed here, only taken from a table entry: its
  // owners wait for partial tiles from later CTAs of the same launch, which
  // assumes the whole persistent grid is resident at once.  A launch that
  // shares the GPU with work on another stream may have CTAs waiting for SMs
  // that its own waiting owners hold, until the bounded wait gives up.  The
  // tail split and the cluster split cover the shapes where it was measured
  // to help, without any wait between CTAs of different clusters.
  return best;
}

// Raster: consecutive units should share the operand that would otherwise be
// re-read from HBM, so walk along N (sharing A tiles) when A is the larger
// operand and along M (sharing B tiles) otherwise.
static int auto_raster(int64_t M, int64_t N, int64_t K) { return M * K > N * K ? 1 : 0; }

static Plan make_plan(int layout, int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in,
                      tg_dtype out, int sms) {
  TableVal v;
  if (table_lookup(TableKey{layout, in, out, M, N, K, batch}, &v)) {
    Plan p;
    p.bn = v.bn;
    p.pair = v.pair != 0;
    p.csplit = v.csplit;
    const int64_t kb = cdiv(K, 64);
    const int64_t tiles = batch * cdiv(M, 128) * cdiv(N, p.bn);
    p.sk = v.splits == 0 && tiles * kb >= 1;
    p.tail = p.sk ? 0 : v.tail;
    const int64_t s = p.sk ? 1 : (v.splits < kb ? v.splits : kb);
    const int64_t kps = cdiv(kb, s);
    p.splits = static_cast<int>(cdiv(kb, kps));
    p.raster_n = v.raster >= 0 ? v.raster : auto_raster(M, N, K);
    p.from_table = true;
    return p;
  }
  Plan p = heuristic_plan(M, N, K, batch, out == TG_F32 ? 4 : 2, sms);
  p.raster_n = auto_raster(M, N, K);
  return p;
}

// CTAs of a stream-K launch (an upper bound for pairs, whose count may be
// capped further by how many clusters fit at once)
static int sk_grid(const Plan& p, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  if (p.pair) {
    const int64_t iters = batch * cdiv(M, 256) * cdiv(N, p.bn) * cdiv(K, 64);
    return 2 * static_cast<int>(iters < sms / 2 ? iters : sms / 2);
  }
  const int64_t iters = batch * cdiv(M, 128) * cdiv(N, p.bn) * cdiv(K, 64);
  return static_cast<int>(iters < sms ? iters : sms);
}

// Tail-split geometry of a plan: a wave is every SM (single CTA) or every
// pair of SMs (256-row tiles)
static TailGeo plan_tail_geo(const Plan& p, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  return tail_geo(M, N, K, batch, p.bn, p.pair ? sms / 2 : sms, p.sk || p.splits > 1 ? 1 : p.tail, p.raster_n,
                  p.pair ? 256 : 128);
}

static size_t plan_ws_bytes(const Plan& p, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  if (p.sk) return sk_ws_bytes(sk_grid(p, M, N, K, batch, sms), p.bn);
  if (p.tail > 1 && p.splits <= 1) return tail_ws_bytes(plan_tail_geo(p, M, N, K, batch, sms));
  return p.splits > 1 ? static_cast<size_t>(p.splits) * batch * M * N * 4 : 0;
}

// Stream-K publication flag value for one launch.  Owners clear the flags
// they consumed, so a workspace that served a completed launch holds zeros; a
// fresh workspace holds arbitrary bytes, which match a 64-bit value that is
// never zero with negligible probability.
static unsigned long long next_epoch() {
  static std::atomic<unsigned long long> ctr{
      (static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) << 20) ^
      0x9E3779B97F4A7C15ull};
  unsigned long long v = ctr.fetch_add(1) + 1;
  return v ? v : ctr.fetch_add(1) + 1;
}

// The deep ring (widths 144 and 192, single CTA) when a CTA streams at least
// 128 K blocks: its epilogues hide behind later MMAs.
static bool plan_deep(const Plan& p, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  if (p.pair || p.csplit > 1 || (p.bn != 192 && p.bn != 144)) return false;
  const int64_t tiles = batch * cdiv(M, 128) * cdiv(N, p.bn);
  const int64_t kb = cdiv(K, 64);
  const int64_t per_cta = p.sk ? cdiv(tiles * kb, sms) : cdiv(tiles * p.splits, sms) * cdiv(kb, p.splits);
  return per_cta >= 128;
}

// "tc nt M=.. N=.. K=.. batch=.. bn=.. [deep|pair|cs] splits=..|sk grid=..
// [tail=AxB|cluster=C] raster=m|n table=hit|miss"
static std::string plan_text(const Plan& p, int layout, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
  const TailGeo tgeo = plan_tail_geo(p, M, N, K, batch, sms);
  char tail[48] = "";
  if (tgeo.tail_tiles > 0) snprintf(tail, sizeof tail, " tail=%dx%d", tgeo.tail_tiles, tgeo.splits);
  if (p.csplit > 1) snprintf(tail, sizeof tail, " cluster=%d", p.csplit);
  char buf[256];
  snprintf(buf, sizeof buf, "tc %s M=%lld N=%lld K=%lld batch=%lld bn=%d%s %s%d%s raster=%c table=%s",
           layout_name(layout), (long long)M, (long long)N, (long long)K, (long long)batch, p.bn,
           plan_deep(p, M, N, K, batch, sms) ? " deep" : (p.pair ? " pair" : (p.csplit > 1 ? " cs" : "")),
           p.sk ? "sk grid=" : "splits=", p.sk ? sk_grid(p, M, N, K, batch, sms) : p.splits, tail,
           p.raster_n ? 'n' : 'm', p.from_table ? "hit" : "miss");
  return buf;
}

// -------------------------------------------------------------- the GEMMs
static bool dtype_in_ok(tg_dtype in) { return in == TG_BF16 || in == TG_F16; }
// the layer products also take FP32 operands (FP32 output only)
static bool dtype_in_ok_layer(tg_dtype in) { return dtype_in_ok(in) || in == TG_F32; }
static bool dtype_out_ok(tg_dtype in, tg_dtype out) { return out == TG_F32 || out == in; }
static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
static size_t dt_bytes(tg_dtype d) { return d == TG_F32 ? 4 : 2; }
static const int64_t kMaxDim = (int64_t(1) << 31) - 1;

struct GemmCall {
  int layout;
  const void* A;
  const void* B;
  void* C;
  int64_t batch, M, N, K;
  int64_t lda, ldb, a_bs, b_bs;  // elements
  tg_dtype in, out;
  int a_kind_override = -1;  // FP32 operand (LoRA dH): CUDA-core path only
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  const char* name;
  int accumulate = 0;  // C += scale * the product (gradient accumulation, LoRA branch added to Y)
  float scale = 1.f;   // without accumulate: C = scale * the product (scaled LoRA gradients)
  int b_kind_override = -1;  // FP32 B operand (an FP32 LoRA factor): CUDA-core path only
};

static bool tc_eligible(const GemmCall& g) {
  if (g.a_kind_override >= 0 || g.b_kind_override >= 0) return false;
  // the tensor-core epilogues neither scale nor add anything but an
  // unscaled FP32 tile (a 16-bit reduce-add would round twice)
  if (g.scale != 1.f || (g.accumulate && g.out != TG_F32)) return false;
  const size_t ob = dt_bytes(g.out);
  return aligned(g.A, 16) && aligned(g.B, 16) && aligned(g.C, 16) && (g.lda * 2) % 16 == 0 &&
         (g.ldb * 2) % 16 == 0 && (g.a_bs * 2) % 16 == 0 && (g.b_bs * 2) % 16 == 0 &&
         (g.N * ob) % 16 == 0 && g.M <= kMaxDim && g.N <= kMaxDim && g.K <= kMaxDim &&
         g.batch <= 65535;
}

// FP32 operands on the tensor cores: each operand cut into three bf16 parts
// in the workspace ([3][elements], parts 8-element aligned), the product run
// over the six part products (reduction 6 K long) on the single-CTA or pair
// kernel (split-K, tail split allowed; a cluster split becomes a split-K).
static bool split3_eligible(const GemmCall& g) {
  return fp32_tc_enabled() && g.in == TG_F32 && g.out == TG_F32 && g.batch == 1 && g.lda % 8 == 0 && g.ldb % 8 == 0 &&
         (g.N * 4) % 16 == 0 && aligned(g.C, 16) && g.M <= kMaxDim && g.N <= kMaxDim && g.K <= kMaxDim / 6 &&
         g.a_kind_override < 0 && g.b_kind_override < 0 && g.scale == 1.f;
}
static int64_t up8(int64_t n) { return (n + 7) / 8 * 8; }
static Plan split3_plan(int layout, int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t kb = (K + 63) / 64;
  Plan p = make_plan(layout, M, N, 6 * kb * 64, 1, TG_F32, TG_F32, sms);
  if (p.csplit > 1) {
    p.splits = p.csplit;
    p.csplit = 0;
  }
  p.sk = false;
  return p;
}
static size_t split3_parts_bytes(int64_t M, int64_t N, int64_t K) {
  return (static_cast<size_t>(3) * (up8(M * K) + up8(N * K)) * 2 + 255) / 256 * 256;
}
static size_t split3_ws_bytes(int layout, int64_t M, int64_t N, int64_t K, int sms) {
  const int64_t kb = (K + 63) / 64;
  return split3_parts_bytes(M, N, K) + plan_ws_bytes(split3_plan(layout, M, N, K, sms), M, N, 6 * kb * 64, 1, sms);
}

static tg_status run_gemm(GemmCall g, DevCtx* ctx) {
  if (g.M == 0 || g.N == 0 || g.batch == 0) {
    record(std::string(g.name) + " empty output: nothing to do");
    return TG_OK;
  }
  const size_t ob = dt_bytes(g.out);
  if (g.K == 0 && g.accumulate) {  // adding an empty sum leaves C as it is
    record(std::string(g.name) + " empty reduction: nothing to add");
    return TG_OK;
  }
  if (g.K == 0) {  // empty sum: zeros (all-zero bits in every output type)
    record(std::string(g.name) + " empty reduction: zero fill");
    return cudaMemsetAsync(g.C, 0, static_cast<size_t>(g.batch * g.M * g.N) * ob, g.stream) == cudaSuccess
               ? TG_OK
               : TG_ERR_CUDA;
  }
  char buf[320];
  if (split3_eligible(g)) {  // FP32 operands: three bf16 parts each, on the tensor cores
    const int64_t na = g.M * g.K, nbb = g.N * g.K, pa = up8(na), pb = up8(nbb);
    const int64_t kb = (g.K + 63) / 64;
    const Plan p = split3_plan(g.layout, g.M, g.N, g.K, ctx->sms);
    const size_t parts = split3_parts_bytes(g.M, g.N, g.K);
    const size_t need = split3_ws_bytes(g.layout, g.M, g.N, g.K, ctx->sms);
    if (g.ws == nullptr || g.ws_bytes < need || !aligned(g.ws, 256)) {
      snprintf(buf, sizeof buf, "%s tc3 %s: workspace %zu bytes needed (256-byte aligned), %zu given", g.name,
               layout_name(g.layout), need, g.ws ? g.ws_bytes : static_cast<size_t>(0));
      record(buf);
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    uint16_t* partsA = static_cast<uint16_t*>(g.ws);
    uint16_t* partsB = partsA + 3 * pa;
    void* pws = static_cast<char*>(g.ws) + parts;
    cudaError_t e = split3_launch(static_cast<const float*>(g.A), na, pa, partsA, g.stream);
    if (e == cudaSuccess) e = split3_launch(static_cast<const float*>(g.B), nbb, pb, partsB, g.stream);
    if (e == cudaSuccess) {
      TcGemm t{};
      t.layout = g.layout;
      t.A = partsA;
      t.B = partsB;
      t.C = g.C;
      t.in_kind = EK_BF16;
      t.out_kind = EK_F32;
      t.batch = 1;
      t.M = g.M;
      t.N = g.N;
      t.K = g.K;
      t.lda = g.lda;
      t.ldb = g.ldb;
      t.a_bstride = pa;
      t.b_bstride = pb;
      t.split3 = 1;
      t.bn = p.bn;
      t.splits = p.splits;
      t.raster_n = p.raster_n;
      t.tail_splits = p.tail;
      t.pair = p.pair ? 1 : 0;
      t.accumulate = g.accumulate;
      t.deep = plan_deep(p, g.M, g.N, 6 * kb * 64, 1, ctx->sms) ? 1 : 0;
      t.ws = pws;
      t.grid = ctx->sms;
      t.stream = g.stream;
      t.status = ctx->status;
      t.timeout_ns = ctx->timeout_ns;
      e = g.layout == LAYOUT_NT ? tc_gemm_launch_nt(t) : g.layout == LAYOUT_NN ? tc_gemm_launch_nn(t) : tc_gemm_launch_tn(t);
      if (e == cudaSuccess && p.splits > 1)
        e = splitk_reduce_launch(static_cast<const float*>(pws), g.C, EK_F32, 1, p.splits, g.M * g.N, g.stream,
                                 g.accumulate);
    }
    std::string txt = plan_text(p, g.layout, g.M, g.N, 6 * kb * 64, 1, ctx->sms);
    if (txt.compare(0, 3, "tc ") == 0) txt = "tc3 " + txt.substr(3);
    record(std::string(g.name) + " " + txt + " " + (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  if (g.in == TG_F32) {  // FP32 operands the tensor-core path cannot take: the CUDA-core FFMA kernel
    FfmaGemm f;
    f.layout = g.layout;
    f.A = static_cast<const float*>(g.A);
    f.B = static_cast<const float*>(g.B);
    f.C = static_cast<float*>(g.C);
    f.M = g.M;
    f.N = g.N;
    f.K = g.K;
    f.lda = g.lda;
    f.ldb = g.ldb;
    f.splits = ffma_splits(g.M, g.N, g.K, ctx->sms);
    f.accumulate = g.accumulate;
    f.stream = g.stream;
    const size_t need = ffma_ws_bytes(g.M, g.N, g.K, ctx->sms);
    if (need > 0 && (g.ws == nullptr || g.ws_bytes < need || !aligned(g.ws, 16))) {
      snprintf(buf, sizeof buf, "%s ffma %s splits=%d: workspace %zu bytes needed, %zu given", g.name,
               layout_name(g.layout), f.splits, need, g.ws ? g.ws_bytes : static_cast<size_t>(0));
      record(buf);
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    f.ws = static_cast<float*>(g.ws);
    cudaError_t e = ffma_gemm_launch(f);
    snprintf(buf, sizeof buf, "%s ffma %s M=%lld N=%lld K=%lld splits=%d %s", g.name, layout_name(g.layout),
             (long long)g.M, (long long)g.N, (long long)g.K, f.splits, e == cudaSuccess ? "ok" : cudaGetErrorString(e));
    record(buf);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  if (tc_eligible(g)) {
    const Plan p = make_plan(g.layout, g.M, g.N, g.K, g.batch, g.in, g.out, ctx->sms);
    const size_t need = plan_ws_bytes(p, g.M, g.N, g.K, g.batch, ctx->sms);
    if (need > 0 && (g.ws == nullptr || g.ws_bytes < need || !aligned(g.ws, 16))) {
      snprintf(buf, sizeof buf, "%s tc %s bn=%d splits=%d: workspace %zu bytes needed, %zu given", g.name,
               layout_name(g.layout), p.bn, p.splits, need, g.ws ? g.ws_bytes : static_cast<size_t>(0));
      record(buf);
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    TcGemm t{};
    t.layout = g.layout;
    t.A = g.A;
    t.B = g.B;
    t.C = g.C;
    t.in_kind = g.in == TG_BF16 ? EK_BF16 : EK_F16;
    t.out_kind = g.out == TG_F32 ? EK_F32 : (g.out == TG_BF16 ? EK_BF16 : EK_F16);
    t.batch = g.batch;
    t.M = g.M;
    t.N = g.N;
    t.K = g.K;
    t.lda = g.lda;
    t.ldb = g.ldb;
    t.a_bstride = g.a_bs;
    t.b_bstride = g.b_bs;
    t.bn = p.bn;
    t.splits = p.splits;
    t.raster_n = p.raster_n;
    t.sk = p.sk ? 1 : 0;
    t.sk_epoch = p.sk ? next_epoch() : 0;
    t.tail_splits = p.tail;
    t.pair = p.pair ? 1 : 0;
    t.csplit = p.csplit;
    t.accumulate = g.accumulate;
    t.deep = plan_deep(p, g.M, g.N, g.K, g.batch, ctx->sms) ? 1 : 0;
    t.ws = g.ws;
    t.grid = ctx->sms;
    t.stream = g.stream;
    t.status = ctx->status;
    t.timeout_ns = ctx->timeout_ns;
    cudaError_t e = g.layout == LAYOUT_NT   ? tc_gemm_launch_nt(t)
                    : g.layout == LAYOUT_NN ? tc_gemm_launch_nn(t)
                                            : tc_gemm_launch_tn(t);
    if (e == cudaSuccess && !p.sk && p.splits > 1)
      e = splitk_reduce_launch(static_cast<const float*>(g.ws), g.C, t.out_kind, g.batch, p.splits, g.M * g.N,
                               g.stream, g.accumulate);
    record(std::string(g.name) + " " + plan_text(p, g.layout, g.M, g.N, g.K, g.batch, ctx->sms) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  // CUDA-core path, same semantics
  SimtGemm s;
  s.A = g.A;
  s.B = g.B;
  s.C = g.C;
  s.a_kind = g.a_kind_override >= 0 ? g.a_kind_override : (g.in == TG_BF16 ? EK_BF16 : EK_F16);
  s.b_kind = g.b_kind_override >= 0 ? g.b_kind_override : (g.in == TG_BF16 ? EK_BF16 : EK_F16);
  s.out_kind = g.out == TG_F32 ? EK_F32 : (g.out == TG_BF16 ? EK_BF16 : EK_F16);
  s.batch = g.batch;
  s.M = g.M;
  s.N = g.N;
  s.K = g.K;
  s.stream = g.stream;
  s.accumulate = g.accumulate;
  s.scale = g.scale;
  s.a_bs = g.a_bs;
  s.b_bs = g.b_bs;
  if (g.layout == LAYOUT_TN) {
    s.a_rs = 1;
    s.a_cs = g.lda;
  } else {
    s.a_rs = g.lda;
    s.a_cs = 1;
  }
  if (g.layout == LAYOUT_NT) {
    s.b_rs = 1;
    s.b_cs = g.ldb;
  } else {
    s.b_rs = g.ldb;
    s.b_cs = 1;
  }
  cudaError_t e = simt_gemm_launch(s);
  snprintf(buf, sizeof buf, "%s simt %s M=%lld N=%lld K=%lld batch=%lld %s", g.name, layout_name(g.layout),
           (long long)g.M, (long long)g.N, (long long)g.K, (long long)g.batch,
           e == cudaSuccess ? "ok" : cudaGetErrorString(e));
  record(buf);
  return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

static size_t gemm_ws_bytes(int layout, int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in, tg_dtype out,
                            int sms) {
  if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return 0;
  if (in == TG_F32) {  // the larger of the tensor-core split's and the FFMA kernel's needs
    if (batch != 1) return 0;
    const size_t a = ffma_ws_bytes(M, N, K, sms), b = K <= kMaxDim / 6 ? split3_ws_bytes(layout, M, N, K, sms) : 0;
    return a > b ? a : b;
  }
  return plan_ws_bytes(make_plan(layout, M, N, K, batch, in, out, sms), M, N, K, batch, sms);
}

// Checks shared by the LoRA and attention products.  Returns TG_OK to proceed.
static tg_status check_common(tg_dtype in, tg_dtype out, std::initializer_list<int64_t> dims) {
  if (!dtype_in_ok(in) || !dtype_out_ok(in, out)) return TG_ERR_UNSUPPORTED_DTYPE;
  for (int64_t d : dims)
    if (d < 0 || d > kMaxDim) return TG_ERR_INVALID_ARG;
  return TG_OK;
}

// The same for the layer products, which also take FP32 operands.
static tg_status check_layer(tg_dtype in, tg_dtype out, std::initializer_list<int64_t> dims) {
  if (!dtype_in_ok_layer(in) || !dtype_out_ok(in, out)) return TG_ERR_UNSUPPORTED_DTYPE;
  for (int64_t d : dims)
    if (d < 0 || d > kMaxDim) return TG_ERR_INVALID_ARG;
  return TG_OK;
}

static tg_status check_ptr(const void* p, int64_t elems, size_t esz) {
  if (elems == 0) return TG_OK;
  if (p == nullptr) return TG_ERR_INVALID_ARG;
  return aligned(p, esz) ? TG_OK : TG_ERR_MISALIGNED;
}

#define TG_TRY(x)                   \
  do {                              \
    tg_status _s = (x);             \
    if (_s != TG_OK) return _s;     \
  } while (0)

}  // namespace tg

using namespace tg;

// =================================================================== C ABI
extern "C" {

int tg_version(void) { return 10000; }

const char* tg_status_string(tg_status s) {
  switch (s) {
    case TG_OK: return "ok";
    case TG_ERR_INVALID_ARG: return "invalid argument";
    case TG_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case TG_ERR_MISALIGNED: return "misaligned pointer";
    case TG_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TG_ERR_CUDA: return "CUDA runtime error";
    case TG_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case TG_ERR_TABLE: return "tile table unreadable";
    case TG_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103";
  }
  return "unknown status";
}

size_t tg_last_call(char* buf, size_t len) {
  const std::string& s = t_last_call;
  if (buf && len) {
    const size_t n = s.size() < len - 1 ? s.size() : len - 1;
    memcpy(buf, s.data(), n);
    buf[n] = '\0';
  }
  return s.size();
}

size_t tg_plan_describe(tg_op op, int64_t M, int64_t N, int64_t K, int64_t batch, tg_dtype in, tg_dtype out,
                        int sms, char* buf, size_t len) {
  if (op != TG_OP_GEMM_FWD && op != TG_OP_GEMM_DGRAD && op != TG_OP_GEMM_WGRAD) return 0;
  if (M <= 0 || N <= 0 || K <= 0 || batch <= 0 || sms < 2 || !dtype_in_ok_layer(in) || !dtype_out_ok(in, out))
    return 0;
  const int layout = op == TG_OP_GEMM_FWD ? LAYOUT_NT : (op == TG_OP_GEMM_DGRAD ? LAYOUT_NN : LAYOUT_TN);
  // contiguous operands: the row pitches the tensor-core path needs
  const int64_t lda = layout == LAYOUT_TN ? M : K, ldb = layout == LAYOUT_NT ? K : N;
  std::string s;
  if (in == TG_F32) {
    if (fp32_tc_enabled() && batch == 1 && lda % 8 == 0 && ldb % 8 == 0 && (N * 4) % 16 == 0 && K <= kMaxDim / 6) {
      // the three-part split on the tensor cores: a reduction six times as long
      const int64_t kb = (K + 63) / 64;
      s = plan_text(split3_plan(layout, M, N, K, sms), layout, M, N, 6 * kb * 64, 1, sms);
      s = "tc3 " + s.substr(3);
    } else {
      s = std::string("ffma ") + layout_name(layout) + " splits=" + std::to_string(ffma_splits(M, N, K, sms));
    }
  } else if ((lda * 2) % 16 || (ldb * 2) % 16 || (N * static_cast<int64_t>(dt_bytes(out))) % 16 || batch > 65535) {
    s = std::string("simt ") + layout_name(layout);
  } else {
    s = plan_text(make_plan(layout, M, N, K, batch, in, out, sms), layout, M, N, K, batch, sms);
  }
  if (buf && len) {
    const size_t n = s.size() < len - 1 ? s.size() : len - 1;
    memcpy(buf, s.data(), n);
    buf[n] = '\0';
  }
  return s.size();
}

tg_status tg_load_table(const char* path) {
  table_env_init();
  return load_table_file(path);
}

tg_status tg_stream_status(void* stream) {
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return TG_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyAsync(&word, ctx->status, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(ctx->status, 0, sizeof word, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return TG_ERR_CUDA;
  return (word & TG_DEVSTAT_TIMEOUT) ? TG_ERR_DEVICE_TIMEOUT : TG_OK;
}

tg_status tg_wait_probe(int64_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000) return TG_ERR_INVALID_ARG;
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaError_t e = wait_probe_launch(static_cast<unsigned long long>(timeout_us) * 1000ull, ctx->status,
                                    static_cast<cudaStream_t>(stream));
  record(std::string("wait_probe ") + (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
  return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

tg_status tg_gemm_fwd(const void* X, const void* W, void* Y, int64_t T, int64_t d_out, int64_t d_in, tg_dtype in,
                      tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_layer(in, out, {T, d_out, d_in}));
  TG_TRY(check_ptr(X, T * d_in, dt_bytes(in)));
  TG_TRY(check_ptr(W, d_out * d_in, dt_bytes(in)));
  TG_TRY(check_ptr(Y, T * d_out, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_NT, X, W, Y, 1, T, d_out, d_in, d_in, d_in, T * d_in, d_out * d_in, in, out, -1, ws, ws_bytes,
             static_cast<cudaStream_t>(stream), "fwd"};
  return run_gemm(g, ctx);
}

tg_status tg_gemm_dgrad(const void* dY, const void* W, void* dX, int64_t T, int64_t d_out, int64_t d_in,
                        tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_layer(in, out, {T, d_out, d_in}));
  TG_TRY(check_ptr(dY, T * d_out, dt_bytes(in)));
  TG_TRY(check_ptr(W, d_out * d_in, dt_bytes(in)));
  TG_TRY(check_ptr(dX, T * d_in, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_NN, dY, W, dX, 1, T, d_in, d_out, d_out, d_in, T * d_out, d_out * d_in, in, out, -1, ws,
             ws_bytes, static_cast<cudaStream_t>(stream), "dgrad"};
  return run_gemm(g, ctx);
}

// ------------------------------------------------ layer product + LoRA branch
// Workspace of a layer product with its LoRA branch added inside the
// product: the staged LoRA block on the tensor-core path; on the CUDA-core
// path an FP32 copy of the output when the output is 16-bit (both products
// are added in FP32 there and the sum rounded once).
static size_t layer_lora_ws(int layout, int64_t M, int64_t N, int64_t K, int64_t r, tg_dtype in, tg_dtype out,
                            int sms) {
  if (r == 0) return gemm_ws_bytes(layout, M, N, K, 1, in, out, sms);  // the plain product
  const size_t tc = lora_block_ws_bytes(M, N);
  const size_t simt = out == TG_F32 ? 0 : static_cast<size_t>(M) * N * 4;
  return tc > simt ? tc : simt;
}

// C[M, N] = A B (layout NT: forward; NN: input gradient) + scale H F, H [M, r]
// (16-bit, or FP32 when h_f32), F: forward B [N, r]; input gradient A [r, N]
static tg_status run_layer_lora(const GemmCall& base, const void* H, int h_f32, const void* F, int64_t r, float scale,
                                DevCtx* ctx) {
  const bool dgrad = base.layout == LAYOUT_NN;
  const int64_t M = base.M, N = base.N;
  if (M == 0 || N == 0) {
    record(std::string(base.name) + " empty output: nothing to do");
    return TG_OK;
  }
  if (r == 0) return run_gemm(base, ctx);
  const int ik = base.in == TG_BF16 ? EK_BF16 : EK_F16;
  const int ok_kind = base.out == TG_F32 ? EK_F32 : ik;
  char buf[320];
  if (tc_eligible(base) && base.K > 0 && r <= 32 && aligned(H, h_f32 ? 4 : 2) && aligned(F, 2)) {
    const size_t need = lora_block_ws_bytes(M, N);
    if (base.ws == nullptr || base.ws_bytes < need || !aligned(base.ws, 16)) {
      snprintf(buf, sizeof buf, "%s: workspace %zu bytes needed, %zu given", base.name, need,
               base.ws ? base.ws_bytes : static_cast<size_t>(0));
      record(buf);
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    // the product's own plan, with every K split undone: the LoRA block is
    // the last K block of each whole tile
    Plan p = make_plan(base.layout, M, N, base.K, 1, base.in, base.out, ctx->sms);
    p.splits = 1;
    p.tail = 0;
    p.sk = false;
    p.csplit = 0;
    const void* A2 = nullptr;
    const void* B2 = nullptr;
    cudaError_t e = lora_block_prep_launch(H, h_f32, F, M, N, r, scale, ik, dgrad ? 1 : 0, base.ws, &A2, &B2, ctx->sms,
                                           base.stream);
    if (e == cudaSuccess) {
      TcGemm t{};
      t.layout = base.layout;
      t.A = base.A;
      t.B = base.B;
      t.C = base.C;
      t.in_kind = ik;
      t.out_kind = ok_kind;
      t.batch = 1;
      t.M = M;
      t.N = N;
      t.K = base.K;
      t.lda = base.lda;
      t.ldb = base.ldb;
      t.a_bstride = base.a_bs;
      t.b_bstride = base.b_bs;
      t.bn = p.bn;
      t.splits = 1;
      t.raster_n = p.raster_n;
      t.pair = p.pair ? 1 : 0;
      t.deep = plan_deep(p, M, N, base.K, 1, ctx->sms) ? 1 : 0;
      t.lora_A2 = A2;
      t.lora_B2 = B2;
      t.grid = ctx->sms;
      t.stream = base.stream;
      t.status = ctx->status;
      t.timeout_ns = ctx->timeout_ns;
      e = dgrad ? tc_gemm_launch_nn(t) : tc_gemm_launch_nt(t);
    }
    record(std::string(base.name) + " " + plan_text(p, base.layout, M, N, base.K, 1, ctx->sms) + " lora r=" +
           std::to_string(r) + " " + (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  // CUDA-core path: both products added in an FP32 buffer (the output itself
  // when it is FP32), then rounded once
  const size_t need = base.out == TG_F32 ? 0 : static_cast<size_t>(M) * N * 4;
  if (need > 0 && (base.ws == nullptr || base.ws_bytes < need || !aligned(base.ws, 16))) {
    snprintf(buf, sizeof buf, "%s simt lora: workspace %zu bytes needed, %zu given", base.name, need,
             base.ws ? base.ws_bytes : static_cast<size_t>(0));
    record(buf);
    return TG_ERR_WORKSPACE_TOO_SMALL;
  }
  void* acc = base.out == TG_F32 ? base.C : base.ws;
  SimtGemm s{};
  s.A = base.A;
  s.B = base.B;
  s.C = acc;
  s.a_kind = ik;
  s.b_kind = ik;
  s.out_kind = EK_F32;
  s.batch = 1;
  s.M = M;
  s.N = N;
  s.K = base.K;
  s.a_bs = base.a_bs;
  s.b_bs = base.b_bs;
  s.a_rs = base.lda;
  s.a_cs = 1;
  if (dgrad) {
    s.b_rs = base.ldb;
    s.b_cs = 1;
  } else {
    s.b_rs = 1;
    s.b_cs = base.ldb;
  }
  s.scale = 1.f;
  s.stream = base.stream;
  cudaError_t e = simt_gemm_launch(s);
  if (e == cudaSuccess) {
    SimtGemm l{};
    l.A = H;
    l.B = F;
    l.C = acc;
    l.a_kind = h_f32 ? EK_F32 : ik;
    l.b_kind = ik;
    l.out_kind = EK_F32;
    l.batch = 1;
    l.M = M;
    l.N = N;
    l.K = r;
    l.a_bs = M * r;
    l.b_bs = N * r;
    l.a_rs = r;
    l.a_cs = 1;
    if (dgrad) {  // F = A [r][N]
      l.b_rs = N;
      l.b_cs = 1;
    } else {  // F = B [N][r]
      l.b_rs = 1;
      l.b_cs = r;
    }
    l.accumulate = 1;
    l.scale = scale;
    l.stream = base.stream;
    e = simt_gemm_launch(l);
  }
  if (e == cudaSuccess && base.out != TG_F32)
    e = splitk_reduce_launch(static_cast<const float*>(acc), base.C, ok_kind, 1, 1, M * N, base.stream, 0);
  snprintf(buf, sizeof buf, "%s simt %s lora M=%lld N=%lld K=%lld r=%lld %s", base.name, layout_name(base.layout),
           (long long)M, (long long)N, (long long)base.K, (long long)r,
           e == cudaSuccess ? "ok" : cudaGetErrorString(e));
  record(buf);
  return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

tg_status tg_gemm_fwd_lora(const void* X, const void* W, const void* H, const void* B, void* Y, int64_t T,
                           int64_t d_out, int64_t d_in, int64_t r, float scale, tg_dtype in, tg_dtype out, void* ws,
                           size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_out, d_in, r}));
  if (!std::isfinite(scale)) return TG_ERR_INVALID_ARG;
  TG_TRY(check_ptr(X, T * d_in, 2));
  TG_TRY(check_ptr(W, d_out * d_in, 2));
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(B, d_out * r, 2));
  TG_TRY(check_ptr(Y, T * d_out, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_NT, X, W, Y, 1, T, d_out, d_in, d_in, d_in, T * d_in, d_out * d_in, in, out, -1, ws, ws_bytes,
             static_cast<cudaStream_t>(stream), "fwd_lora"};
  return run_layer_lora(g, H, 0, B, r, scale, ctx);
}

tg_status tg_gemm_dgrad_lora(const void* dY, const void* W, const float* dH, const void* A, void* dX, int64_t T,
                             int64_t d_out, int64_t d_in, int64_t r, float scale, tg_dtype in, tg_dtype out, void* ws,
                             size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_out, d_in, r}));
  if (!std::isfinite(scale)) return TG_ERR_INVALID_ARG;
  TG_TRY(check_ptr(dY, T * d_out, 2));
  TG_TRY(check_ptr(W, d_out * d_in, 2));
  TG_TRY(check_ptr(dH, T * r, 4));
  TG_TRY(check_ptr(A, r * d_in, 2));
  TG_TRY(check_ptr(dX, T * d_in, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_NN, dY, W, dX, 1, T, d_in, d_out, d_out, d_in, T * d_out, d_out * d_in, in, out, -1, ws,
             ws_bytes, static_cast<cudaStream_t>(stream), "dgrad_lora"};
  return run_layer_lora(g, dH, 1, A, r, scale, ctx);
}

tg_status tg_gemm_wgrad(const void* dY, const void* X, void* dW, int64_t T, int64_t d_out, int64_t d_in,
                        tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_layer(in, out, {T, d_out, d_in}));
  TG_TRY(check_ptr(dY, T * d_out, dt_bytes(in)));
  TG_TRY(check_ptr(X, T * d_in, dt_bytes(in)));
  TG_TRY(check_ptr(dW, d_out * d_in, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_TN, dY, X, dW, 1, d_out, d_in, T, d_out, d_in, T * d_out, T * d_in, in, out, -1, ws,
             ws_bytes, static_cast<cudaStream_t>(stream), "wgrad"};
  return run_gemm(g, ctx);
}

tg_status tg_gemm_wgrad_accumulate(const void* dY, const void* X, float* dW, int64_t T, int64_t d_out,
                                   int64_t d_in, tg_dtype in, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_layer(in, TG_F32, {T, d_out, d_in}));
  TG_TRY(check_ptr(dY, T * d_out, dt_bytes(in)));
  TG_TRY(check_ptr(X, T * d_in, dt_bytes(in)));
  TG_TRY(check_ptr(dW, d_out * d_in, 4));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  GemmCall g{LAYOUT_TN, dY, X, dW, 1, d_out, d_in, T, d_out, d_in, T * d_out, T * d_in, in, TG_F32, -1, ws,
             ws_bytes, static_cast<cudaStream_t>(stream), "wgrad_accumulate", 1};
  return run_gemm(g, ctx);
}

// ------------------------------------------------------------- attention
static bool attn_call(tg_attn_op op, const void* A, const void* B, void* C, int64_t batch, int64_t s, int64_t d,
                      tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream, GemmCall* g) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (op) {
    case TG_ATTN_QK:
    case TG_ATTN_DO_VT:  // [s,d] x [s,d]^T -> [s,s]
      *g = GemmCall{LAYOUT_NT, A, B, C, batch, s, s, d, d, d, s * d, s * d, in, out, -1, ws, ws_bytes, st,
                    op == TG_ATTN_QK ? "attn_qk" : "attn_do_vt"};
      return true;
    case TG_ATTN_PV:
    case TG_ATTN_DS_K:  // [s,s] x [s,d] -> [s,d]
      *g = GemmCall{LAYOUT_NN, A, B, C, batch, s, d, s, s, d, s * s, s * d, in, out, -1, ws, ws_bytes, st,
                    op == TG_ATTN_PV ? "attn_pv" : "attn_ds_k"};
      return true;
    case TG_ATTN_PT_DO:
    case TG_ATTN_DST_Q:  // [s,s]^T x [s,d] -> [s,d]
      *g = GemmCall{LAYOUT_TN, A, B, C, batch, s, d, s, s, d, s * s, s * d, in, out, -1, ws, ws_bytes, st,
                    op == TG_ATTN_PT_DO ? "attn_pt_do" : "attn_dst_q"};
      return true;
  }
  return false;
}

tg_status tg_bmm_attn(tg_attn_op op, const void* A, const void* B, void* C, int64_t batch, int64_t s, int64_t d,
                      tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {batch, s, d}));
  GemmCall g;
  if (!attn_call(op, A, B, C, batch, s, d, in, out, ws, ws_bytes, stream, &g)) return TG_ERR_INVALID_ARG;
  const bool ss_a = op == TG_ATTN_PV || op == TG_ATTN_DS_K || op == TG_ATTN_PT_DO || op == TG_ATTN_DST_Q;
  const bool ss_c = op == TG_ATTN_QK || op == TG_ATTN_DO_VT;
  TG_TRY(check_ptr(A, batch * s * (ss_a ? s : d), 2));
  TG_TRY(check_ptr(B, batch * s * d, 2));
  TG_TRY(check_ptr(C, batch * s * (ss_c ? s : d), dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  return run_gemm(g, ctx);
}

// ------------------------------------------------------------------ LoRA
// Rank 16 with 16-byte-aligned rows takes the streaming kernels (lora.cu);
// anything else is composed from the general products.
static bool lora_stream_ok(int64_t r, std::initializer_list<int64_t> widths,
                           std::initializer_list<const void*> ptrs16) {
  if (r != 16) return false;
  for (int64_t w : widths)
    if (w % 8 != 0 || w > (int64_t(1) << 30)) return false;
  for (const void* p : ptrs16)
    if (p != nullptr && !aligned(p, 16)) return false;
  return true;
}

tg_status tg_lora_down(const void* X, const void* A, void* H, int64_t T, int64_t d_in, int64_t r, tg_dtype in,
                       tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_in, r}));
  TG_TRY(check_ptr(X, T * d_in, 2));
  TG_TRY(check_ptr(A, r * d_in, 2));
  TG_TRY(check_ptr(H, T * r, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_in > 0 && lora_stream_ok(r, {d_in}, {X, A})) {
    LoraArgs a{};
    a.X = X;
    a.A = A;
    a.out = H;
    a.T = T;
    a.d_in = d_in;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    cudaError_t e = lora_down_launch(a);
    record(std::string("lora_down stream T=") + std::to_string(T) + " d_in=" + std::to_string(d_in) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  GemmCall g{LAYOUT_NT, X, A, H, 1, T, r, d_in, d_in, d_in, T * d_in, r * d_in, in, out, -1, ws, ws_bytes, st,
             "lora_down"};
  return run_gemm(g, ctx);
}

tg_status tg_lora_up(const void* H, const void* B, void* Y, int64_t T, int64_t d_out, int64_t r, tg_dtype in,
                     tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_out, r}));
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(B, d_out * r, 2));
  TG_TRY(check_ptr(Y, T * d_out, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_out > 0 && lora_stream_ok(r, {d_out}, {H, B, Y})) {
    LoraArgs a{};
    a.H = H;
    a.B = B;
    a.out = Y;
    a.T = T;
    a.d_out = d_out;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    cudaError_t e = lora_up_launch(a);
    record(std::string("lora_up stream T=") + std::to_string(T) + " d_out=" + std::to_string(d_out) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  GemmCall g{LAYOUT_NT, H, B, Y, 1, T, d_out, r, r, r, T * r, d_out * r, in, out, -1, ws, ws_bytes, st,
             "lora_up"};
  return run_gemm(g, ctx);
}

tg_status tg_lora_up_add(const void* H, const void* B, void* Y, int64_t T, int64_t d_out, int64_t r, float scale,
                         tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_out, r}));
  if (!std::isfinite(scale)) return TG_ERR_INVALID_ARG;
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(B, d_out * r, 2));
  TG_TRY(check_ptr(Y, T * d_out, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_out > 0 && lora_stream_ok(r, {d_out}, {H, B, Y})) {
    LoraArgs a{};
    a.H = H;
    a.B = B;
    a.out = Y;
    a.T = T;
    a.d_out = d_out;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    a.add = 1;
    a.scale = scale;
    cudaError_t e = lora_up_launch(a);
    record(std::string("lora_up_add stream T=") + std::to_string(T) + " d_out=" + std::to_string(d_out) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  GemmCall g{LAYOUT_NT, H, B, Y, 1, T, d_out, r, r, r, T * r, d_out * r, in, out, -1, ws, ws_bytes, st,
             "lora_up_add", 1, scale};
  return run_gemm(g, ctx);
}

// workspace of the composed LoRA gradient: [dH f32 (if not given)] [sub-GEMM ws]
static size_t lora_grad_generic_ws(int64_t T, int64_t d_in, int64_t d_out, int64_t r, tg_dtype in, tg_dtype out,
                                   int sms) {
  // dH = dY . B and dB = dY^T . H run one after the other and share the space
  const size_t a = gemm_ws_bytes(LAYOUT_NN, T, r, d_out, 1, in, TG_F32, sms);
  const size_t b = gemm_ws_bytes(LAYOUT_TN, d_out, r, T, 1, in, out, sms);
  (void)d_in;
  const size_t dh = (static_cast<size_t>(T * r * 4) + 255) / 256 * 256;
  return dh + (a > b ? a : b);
}

// add = 0: the plain gradients; add = 1: dX += scale dH A, dA and dB scaled
static tg_status lora_grad_impl(const void* X, const void* A, const void* B, const void* H, const void* dY, void* dA,
                                void* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in, int64_t d_out, int64_t r,
                                tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream, int add,
                                float scale) {
  const std::string name = add ? "lora_grad_add" : "lora_grad";
  TG_TRY(check_common(in, out, {T, d_in, d_out, r}));
  if (!std::isfinite(scale)) return TG_ERR_INVALID_ARG;
  TG_TRY(check_ptr(X, T * d_in, 2));
  TG_TRY(check_ptr(A, r * d_in, 2));
  TG_TRY(check_ptr(B, d_out * r, 2));
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(dY, T * d_out, 2));
  TG_TRY(check_ptr(dA, r * d_in, dt_bytes(out)));
  TG_TRY(check_ptr(dB, d_out * r, dt_bytes(out)));
  TG_TRY(check_ptr(dX, T * d_in, dt_bytes(out)));
  if (dH_f32 && !aligned(dH_f32, 4)) return TG_ERR_MISALIGNED;
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_in > 0 && d_out > 0 && lora_stream_ok(r, {d_in, d_out}, {X, B, dY, dX, dH_f32, H})) {
    const size_t need = lora_grad_ws_bytes(T, d_in, d_out, r, ctx->sms);
    if (ws == nullptr || ws_bytes < need || !aligned(ws, 256)) {
      record(name + " stream: workspace too small");
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    LoraArgs a{};
    a.X = X;
    a.A = A;
    a.B = B;
    a.H = H;
    a.dY = dY;
    a.out = dA;
    a.out2 = dB;
    a.out3 = dX;
    a.out4 = dH_f32;
    a.ws = static_cast<float*>(ws);
    a.T = T;
    a.d_in = d_in;
    a.d_out = d_out;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    a.add = add;
    a.scale = scale;
    cudaError_t e = lora_grad_launch(a);
    record(name + " stream T=" + std::to_string(T) + " d_in=" + std::to_string(d_in) +
           " d_out=" + std::to_string(d_out) + " " + (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  // general composition (any rank, any alignment)
  const size_t dh_bytes = dH_f32 ? 0 : (static_cast<size_t>(T * r * 4) + 255) / 256 * 256;
  const size_t total = lora_grad_generic_ws(T, d_in, d_out, r, in, out, ctx->sms);
  const size_t sub = total - (static_cast<size_t>(T * r * 4) + 255) / 256 * 256;
  if (dh_bytes + sub > 0 && (ws == nullptr || ws_bytes < dh_bytes + sub || !aligned(ws, 256)))
    return TG_ERR_WORKSPACE_TOO_SMALL;
  float* dH = dH_f32 ? dH_f32 : static_cast<float*>(ws);
  void* sub_ws = static_cast<char*>(ws) + dh_bytes;
  // dH = dY . B (FP32)
  GemmCall g1{LAYOUT_NN, dY, B, dH, 1, T, r, d_out, d_out, r, T * d_out, d_out * r, in, TG_F32, -1, sub_ws, sub,
              st, "lora_grad.dH"};
  TG_TRY(run_gemm(g1, ctx));
  // dB = dY^T . H  (scaled)
  GemmCall g2{LAYOUT_TN, dY, H, dB, 1, d_out, r, T, d_out, r, T * d_out, T * r, in, out, -1, sub_ws, sub, st,
              add ? "lora_grad_add.dB" : "lora_grad.dB", 0, add ? scale : 1.f};
  TG_TRY(run_gemm(g2, ctx));
  // dA = dH^T . X (scaled)  and  dX = dH . A (or dX += scale dH . A)  with the FP32 dH operand
  GemmCall g3{LAYOUT_TN, dH, X, dA, 1, r, d_in, T, r, d_in, T * r, T * d_in, in, out, EK_F32, nullptr, 0, st,
              add ? "lora_grad_add.dA" : "lora_grad.dA", 0, add ? scale : 1.f};
  TG_TRY(run_gemm(g3, ctx));
  GemmCall g4{LAYOUT_NN, dH, A, dX, 1, T, d_in, r, r, d_in, T * r, r * d_in, in, out, EK_F32, nullptr, 0, st,
              add ? "lora_grad_add.dX" : "lora_grad.dX", add, add ? scale : 1.f};
  return run_gemm(g4, ctx);
}

tg_status tg_lora_grad(const void* X, const void* A, const void* B, const void* H, const void* dY, void* dA,
                       void* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in, int64_t d_out, int64_t r,
                       tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  return lora_grad_impl(X, A, B, H, dY, dA, dB, dX, dH_f32, T, d_in, d_out, r, in, out, ws, ws_bytes, stream, 0,
                        1.f);
}

tg_status tg_lora_grad_add(const void* X, const void* A, const void* B, const void* H, const void* dY, void* dA,
                           void* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in, int64_t d_out, int64_t r,
                           float scale, tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  return lora_grad_impl(X, A, B, H, dY, dA, dB, dX, dH_f32, T, d_in, d_out, r, in, out, ws, ws_bytes, stream, 1,
                        scale);
}

// ---- LoRA with FP32 factors (the factors as an optimizer keeps them; activations 16-bit)

static size_t w32_generic_grad_ws(int64_t T, int64_t d_in, int64_t d_out, int64_t r, tg_dtype in, int sms) {
  // dH = dY . B (FP32, CUDA cores) and dB = dY^T . H (FP32 out) run one after the other
  const size_t b = gemm_ws_bytes(LAYOUT_TN, d_out, r, T, 1, in, TG_F32, sms);
  (void)d_in;
  return (static_cast<size_t>(T * r * 4) + 255) / 256 * 256 + b;
}

static size_t w32_ws(int which, int64_t T, int64_t d_in, int64_t d_out, int64_t r, tg_dtype in, int sms) {
  const size_t stream = r == 16 ? lora_w32_ws_bytes(which, T, d_in, d_out, sms) : 0;
  const size_t generic = which == 2 ? w32_generic_grad_ws(T, d_in, d_out, r, in, sms) : 0;
  return stream > generic ? stream : generic;
}

tg_status tg_lora_down_f32w(const void* X, const float* A, void* H, int64_t T, int64_t d_in, int64_t r, tg_dtype in,
                            tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_in, r}));
  TG_TRY(check_ptr(X, T * d_in, 2));
  TG_TRY(check_ptr(A, r * d_in, 4));
  TG_TRY(check_ptr(H, T * r, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_in > 0 && lora_stream_ok(r, {d_in}, {X})) {
    const size_t need = lora_w32_ws_bytes(0, T, d_in, 0, ctx->sms);
    if (ws == nullptr || ws_bytes < need || !aligned(ws, 256)) {
      record("lora_down_f32w stream: workspace too small");
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    LoraArgs a{};
    a.X = X;
    a.A = A;
    a.out = H;
    a.ws = static_cast<float*>(ws);
    a.T = T;
    a.d_in = d_in;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    a.w32 = 1;
    cudaError_t e = lora_down_launch(a);
    record(std::string("lora_down_f32w stream T=") + std::to_string(T) + " d_in=" + std::to_string(d_in) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  GemmCall g{LAYOUT_NT, X, A, H, 1, T, r, d_in, d_in, d_in, T * d_in, r * d_in, in, out, -1, nullptr, 0, st,
             "lora_down_f32w"};
  g.b_kind_override = EK_F32;
  return run_gemm(g, ctx);
}

tg_status tg_lora_up_f32w(const void* H, const float* B, void* Y, int64_t T, int64_t d_out, int64_t r, tg_dtype in,
                          tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_out, r}));
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(B, d_out * r, 4));
  TG_TRY(check_ptr(Y, T * d_out, dt_bytes(out)));
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_out > 0 && lora_stream_ok(r, {d_out}, {H, Y, B})) {  // B: 16-byte loads of FP32 rows
    const size_t need = lora_w32_ws_bytes(1, T, 0, d_out, ctx->sms);
    if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 256))) {
      record("lora_up_f32w stream: workspace too small");
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    LoraArgs a{};
    a.H = H;
    a.B = B;
    a.out = Y;
    a.ws = static_cast<float*>(ws);
    a.T = T;
    a.d_out = d_out;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    a.w32 = 1;
    cudaError_t e = lora_up_launch(a);
    record(std::string("lora_up_f32w stream T=") + std::to_string(T) + " d_out=" + std::to_string(d_out) + " " +
           (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  GemmCall g{LAYOUT_NT, H, B, Y, 1, T, d_out, r, r, r, T * r, d_out * r, in, out, -1, nullptr, 0, st,
             "lora_up_f32w"};
  g.b_kind_override = EK_F32;
  return run_gemm(g, ctx);
}

tg_status tg_lora_grad_f32w(const void* X, const float* A, const float* B, const void* H, const void* dY, float* dA,
                            float* dB, void* dX, float* dH_f32, int64_t T, int64_t d_in, int64_t d_out, int64_t r,
                            tg_dtype in, tg_dtype out, void* ws, size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {T, d_in, d_out, r}));
  TG_TRY(check_ptr(X, T * d_in, 2));
  TG_TRY(check_ptr(A, r * d_in, 4));
  TG_TRY(check_ptr(B, d_out * r, 4));
  TG_TRY(check_ptr(H, T * r, 2));
  TG_TRY(check_ptr(dY, T * d_out, 2));
  TG_TRY(check_ptr(dA, r * d_in, 4));
  TG_TRY(check_ptr(dB, d_out * r, 4));
  TG_TRY(check_ptr(dX, T * d_in, dt_bytes(out)));
  if (dH_f32 && !aligned(dH_f32, 4)) return TG_ERR_MISALIGNED;
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T > 0 && d_in > 0 && d_out > 0 && lora_stream_ok(r, {d_in, d_out}, {X, dY, dX, dH_f32, H})) {
    const size_t need = lora_w32_ws_bytes(2, T, d_in, d_out, ctx->sms);
    if (ws == nullptr || ws_bytes < need || !aligned(ws, 256)) {
      record("lora_grad_f32w stream: workspace too small");
      return TG_ERR_WORKSPACE_TOO_SMALL;
    }
    LoraArgs a{};
    a.X = X;
    a.A = A;
    a.B = B;
    a.H = H;
    a.dY = dY;
    a.out = dA;
    a.out2 = dB;
    a.out3 = dX;
    a.out4 = dH_f32;
    a.ws = static_cast<float*>(ws);
    a.T = T;
    a.d_in = d_in;
    a.d_out = d_out;
    a.r = r;
    a.in_kind = in == TG_BF16 ? EK_BF16 : EK_F16;
    a.out_kind = out == TG_F32 ? EK_F32 : a.in_kind;
    a.num_sms = ctx->sms;
    a.stream = st;
    a.status = ctx->status;
    a.timeout_ns = ctx->timeout_ns;
    a.scale = 1.f;
    a.w32 = 1;
    cudaError_t e = lora_grad_launch(a);
    record(std::string("lora_grad_f32w stream T=") + std::to_string(T) + " d_in=" + std::to_string(d_in) +
           " d_out=" + std::to_string(d_out) + " " + (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
  }
  // general composition on the CUDA cores for the FP32 factor operands
  const size_t dh_bytes = dH_f32 ? 0 : (static_cast<size_t>(T * r * 4) + 255) / 256 * 256;
  const size_t total = w32_generic_grad_ws(T, d_in, d_out, r, in, ctx->sms);
  const size_t sub = total - (static_cast<size_t>(T * r * 4) + 255) / 256 * 256;
  if (dh_bytes + sub > 0 && (ws == nullptr || ws_bytes < dh_bytes + sub || !aligned(ws, 256)))
    return TG_ERR_WORKSPACE_TOO_SMALL;
  float* dH = dH_f32 ? dH_f32 : static_cast<float*>(ws);
  void* sub_ws = static_cast<char*>(ws) + dh_bytes;
  // dH = dY . B (FP32)
  GemmCall g1{LAYOUT_NN, dY, B, dH, 1, T, r, d_out, d_out, r, T * d_out, d_out * r, in, TG_F32, -1, nullptr, 0, st,
              "lora_grad_f32w.dH"};
  g1.b_kind_override = EK_F32;
  TG_TRY(run_gemm(g1, ctx));
  // dB = dY^T . H (FP32)
  GemmCall g2{LAYOUT_TN, dY, H, dB, 1, d_out, r, T, d_out, r, T * d_out, T * r, in, TG_F32, -1, sub_ws, sub, st,
              "lora_grad_f32w.dB"};
  TG_TRY(run_gemm(g2, ctx));
  // dA = dH^T . X (FP32)  and  dX = dH . A
  GemmCall g3{LAYOUT_TN, dH, X, dA, 1, r, d_in, T, r, d_in, T * r, T * d_in, in, TG_F32, EK_F32, nullptr, 0, st,
              "lora_grad_f32w.dA"};
  TG_TRY(run_gemm(g3, ctx));
  GemmCall g4{LAYOUT_NN, dH, A, dX, 1, T, d_in, r, r, d_in, T * r, r * d_in, in, out, EK_F32, nullptr, 0, st,
              "lora_grad_f32w.dX"};
  g4.b_kind_override = EK_F32;
  return run_gemm(g4, ctx);
}

tg_status tg_attn_fwd(const void* Q, const void* K, const void* V, void* O, int64_t heads, int64_t s, int64_t d,
                      float scale, tg_dtype in, tg_dtype out, void* stream) {
  TG_TRY(check_common(in, out, {heads, s, d}));
  if (d != 64 || !std::isfinite(scale) || heads > 65535) return TG_ERR_INVALID_ARG;
  const int64_t n = heads * s * d;
  TG_TRY(check_ptr(Q, n, 2));
  TG_TRY(check_ptr(K, n, 2));
  TG_TRY(check_ptr(V, n, 2));
  TG_TRY(check_ptr(O, n, dt_bytes(out)));
  if (n > 0 && !(aligned(Q, 16) && aligned(K, 16) && aligned(V, 16) && aligned(O, 16))) return TG_ERR_MISALIGNED;
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  const int ik = in == TG_BF16 ? EK_BF16 : EK_F16;
  const int ok = out == TG_F32 ? EK_F32 : ik;
  cudaError_t e = attn_fwd_tc_launch(Q, K, V, O, heads, s, d, scale, ik, ok, ctx->status, ctx->timeout_ns,
                                     static_cast<cudaStream_t>(stream));
  record(std::string("attn_fwd fused tc heads=") + std::to_string(heads) + " s=" + std::to_string(s) + " " +
         (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
  return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

tg_status tg_attn_bwd(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                      int64_t heads, int64_t s, int64_t d, float scale, tg_dtype in, tg_dtype out, void* ws,
                      size_t ws_bytes, void* stream) {
  TG_TRY(check_common(in, out, {heads, s, d}));
  if (d != 64 || !std::isfinite(scale) || heads > 65535) return TG_ERR_INVALID_ARG;
  const int64_t n = heads * s * d;
  TG_TRY(check_ptr(Q, n, 2));
  TG_TRY(check_ptr(K, n, 2));
  TG_TRY(check_ptr(V, n, 2));
  TG_TRY(check_ptr(dO, n, 2));
  TG_TRY(check_ptr(dQ, n, dt_bytes(out)));
  TG_TRY(check_ptr(dK, n, dt_bytes(out)));
  TG_TRY(check_ptr(dV, n, dt_bytes(out)));
  if (n > 0 && !(aligned(Q, 16) && aligned(K, 16) && aligned(V, 16) && aligned(dO, 16) && aligned(dQ, 16) &&
                 aligned(dK, 16) && aligned(dV, 16)))
    return TG_ERR_MISALIGNED;
  const size_t need = n > 0 ? attn_bwd_ws_bytes(heads, s) : 0;
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return TG_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned(ws, 16)) return TG_ERR_MISALIGNED;
  DevCtx* ctx = nullptr;
  TG_TRY(device_ctx(&ctx));
  const int ik = in == TG_BF16 ? EK_BF16 : EK_F16;
  const int ok = out == TG_F32 ? EK_F32 : ik;
  cudaError_t e = attn_bwd_tc_launch(Q, K, V, dO, dQ, dK, dV, heads, s, d, scale, ik, ok, ws, ctx->status,
                                     ctx->timeout_ns, static_cast<cudaStream_t>(stream));
  record(std::string("attn_bwd fused tc heads=") + std::to_string(heads) + " s=" + std::to_string(s) + " " +
         (e == cudaSuccess ? "ok" : cudaGetErrorString(e)));
  return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

size_t tg_workspace_size(tg_op op, int64_t d0, int64_t d1, int64_t d2, int64_t d3, tg_dtype in, tg_dtype out) {
  const bool layer = op == TG_OP_GEMM_FWD || op == TG_OP_GEMM_DGRAD || op == TG_OP_GEMM_WGRAD;
  if (!(layer ? dtype_in_ok_layer(in) : dtype_in_ok(in)) || !dtype_out_ok(in, out)) return SIZE_MAX;
  if (d0 < 0 || d1 < 0 || d2 < 0 || d3 < 0) return SIZE_MAX;
  DevCtx* ctx = nullptr;
  if (device_ctx(&ctx) != TG_OK) return SIZE_MAX;
  switch (op) {
    case TG_OP_GEMM_FWD: return gemm_ws_bytes(LAYOUT_NT, d0, d1, d2, 1, in, out, ctx->sms);
    case TG_OP_GEMM_DGRAD: return gemm_ws_bytes(LAYOUT_NN, d0, d2, d1, 1, in, out, ctx->sms);
    case TG_OP_GEMM_WGRAD: return gemm_ws_bytes(LAYOUT_TN, d1, d2, d0, 1, in, out, ctx->sms);
    // LoRA: the larger of the streaming and the general requirement (the
    // choice between them also depends on pointer alignment)
    case TG_OP_LORA_DOWN: return gemm_ws_bytes(LAYOUT_NT, d0, d2, d1, 1, in, out, ctx->sms);
    case TG_OP_LORA_UP: return gemm_ws_bytes(LAYOUT_NT, d0, d1, d2, 1, in, out, ctx->sms);
    case TG_OP_LORA_GRAD: {
      const size_t a = lora_grad_generic_ws(d0, d1, d2, d3, in, out, ctx->sms);
      const size_t b = d3 == 16 ? lora_grad_ws_bytes(d0, d1, d2, d3, ctx->sms) : 0;
      return a > b ? a : b;
    }
    case TG_OP_LORA_DOWN_F32W: return w32_ws(0, d0, d1, 0, d2, in, ctx->sms);
    case TG_OP_LORA_UP_F32W: return w32_ws(1, d0, 0, d1, d2, in, ctx->sms);
    case TG_OP_LORA_GRAD_F32W: return w32_ws(2, d0, d1, d2, d3, in, ctx->sms);
    case TG_OP_ATTN_BWD: return d2 == 64 ? attn_bwd_ws_bytes(d0, d1) : SIZE_MAX;
    case TG_OP_GEMM_FWD_LORA: return layer_lora_ws(LAYOUT_NT, d0, d1, d2, d3, in, out, ctx->sms);
    case TG_OP_GEMM_DGRAD_LORA: return layer_lora_ws(LAYOUT_NN, d0, d2, d1, d3, in, out, ctx->sms);
    case TG_OP_BMM_ATTN: {
      GemmCall g;
      if (!attn_call(static_cast<tg_attn_op>(d0), nullptr, nullptr, nullptr, d1, d2, d3, in, out, nullptr, 0,
                     nullptr, &g))
        return SIZE_MAX;
      return gemm_ws_bytes(g.layout, g.M, g.N, g.K, g.batch, in, out, ctx->sms);
    }
  }
  return SIZE_MAX;
}

}  // extern "C"
