// fa_api.cu — host side of the C ABI declared in include/fa.h: argument
// validation, device checks, TMA tensor-map encoding, kernel dispatch and the
// per-device status word.  Nothing here computes attention; every step of the
// forward runs in the kernels of fa_tc_*.cu and fa_simt.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mu;
unsigned *g_status[kMaxDevices] = {};   // device status word per device
int g_dev_ok[kMaxDevices] = {};         // 0 unknown, 1 sm_103, -1 other
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<int> g_skip_v_load{0};
std::atomic<unsigned long long> g_wait_limit_ns{0};
std::atomic<int> g_force_ctas{0};   // persistent grid size forced by a test (0 = automatic)
std::atomic<int> g_force_group{0};  // planes per group forced by a test (0 = automatic)
std::atomic<int> g_force_block{0};  // blocked schedule forced by a test (0 = automatic)
std::atomic<long long> g_dbg_lse_shrink{0};  // debug build: LSE extent understated by a test

size_t elem_size(int dtype) { return (dtype == FA_DTYPE_BF16 || dtype == FA_DTYPE_F16) ? 2 : 4; }

bool overlap(const void *a, size_t an, const void *b, size_t bn) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// Host-side checks shared by fa_fwd and fa_fwd_host.
int validate(const void *q, const void *k, const void *v, const void *o, const float *lse,
             int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  // The kernels index (batch, head) planes with 32-bit ints (b * H + h).
  if (static_cast<long long>(B) * H > 2147483647LL) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_F32_SIMT &&
      dtype != FA_DTYPE_F16)
    return FA_ERR_INVALID_ARG;
  for (const void *ptr : {q, k, v, o})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0) return FA_ERR_INVALID_ARG;
  // Sizes: every flat index must fit comfortably in 63 bits and the TMA
  // coordinates in 31 bits.
  const double rows_q = static_cast<double>(B) * H * Nq, rows_k = static_cast<double>(B) * H * Nk;
  if (rows_q * d >= 9.0e18 || rows_k * d >= 9.0e18) return FA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t qn = static_cast<size_t>(B) * H * Nq * d * es;
  const size_t kn = static_cast<size_t>(B) * H * Nk * d * es;
  const size_t ln = static_cast<size_t>(B) * H * Nq * sizeof(float);
  if (overlap(o, qn, q, qn) || overlap(o, qn, k, kn) || overlap(o, qn, v, kn) ||
      overlap(o, qn, lse, ln) || overlap(lse, ln, q, qn) || overlap(lse, ln, k, kn) ||
      overlap(lse, ln, v, kn))
    return FA_ERR_INVALID_ARG;
  // The compiled set of kernels.
  if ((dtype == FA_DTYPE_BF16 || dtype == FA_DTYPE_F16) && d != 32 && d != 64 && d != 128 &&
      d != 256)
    return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_F32 && d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_F32_SIMT && d > 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// FA_OK when device `dev` is an sm_103 (the only code compiled in), else
// FA_ERR_UNSUPPORTED; the answer is cached per device.  Called with g_mu held.
int check_sm103(int dev) {
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_dev_ok[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED;
}

// The current device must be sm_103; also makes sure its status word exists.
// Returns FA_OK and the status pointer.
int device_setup(unsigned **status) {
  int rc, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if ((rc = check_sm103(dev)) != FA_OK) return rc;
  if (g_status[dev] == nullptr) {
    unsigned *ptr = nullptr;
    if (cudaMalloc(&ptr, 256) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaMemset(ptr, 0, 256) != cudaSuccess) {
      cudaFree(ptr);
      return FA_ERR_CUDA;
    }
    g_status[dev] = ptr;
  }
  *status = g_status[dev];
  return FA_OK;
}

int get_encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode) return FA_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult qres = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || fn == nullptr)
    return FA_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return FA_OK;
}

// 3-D view [B*H, N, d] of a [B, H, N, d] tensor, boxes of {128 bytes of d,
// 128 rows, 1 head}, 128-byte swizzle, zero fill outside the tensor (rows past
// N read as zeros and are clipped on store).
int encode_map(CUtensorMap *map, const void *base, int dtype, int BH, int N, int d) {
  const CUtensorMapDataType dt = dtype == FA_DTYPE_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t es = elem_size(dtype);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es,
                           static_cast<cuuint64_t>(d) * static_cast<cuuint64_t>(N) * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(fa::BM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int sm_count();

// K and V bytes of the planes that run at the same time in a persistent grid
// (one group of fwd_item): sized to stay in L2 (129 MB on GB300) next to the
// Q tiles and O stores passing through, so each head's K/V tiles come from
// HBM about once while all of its query tiles run.
constexpr double kL2GroupBytes = 48.0 * (1 << 20);

// Blocked schedule: items per CTA G in {1, 2, 4} for the one-tile kernel.
// A CTA's fixed cost (set-up, pipeline fill, its last epilogue) is paid once
// for its G items, each next item's loads and first products overlap the
// previous epilogue, and with G >= 2 the zigzag order gives every causal
// CTA the same work; but fewer, longer CTAs can leave the SMs' last wave part
// empty.  G minimises a makespan model in units of one key tile's time t:
//   G >= 2: ceil(CTAs / SMs) * (G * nbar + c)          (equal CTAs)
//   G = 1:  CTAs * (nbar + c1) / SMs + nbar             (causal: uneven CTAs,
//           heaviest first; non-causal: as G >= 2 with c1)
// nbar = mean key tiles per query tile; c and c1 = fixed cost per CTA with
// and without a following item to hide the epilogue.  Fitted on GB300 at
// d = 128 (t = 0.77 us, c = 2.0 us, c1 = 3.0 us); a tile's time scales with
// the head dim, the fixed cost does not.  A G that leaves fewer CTAs than
// SMs is not taken.
int blocked_items(int d, int causal, long long planes, int n_qtiles, int n_ktiles, int num_sms) {
  if (n_qtiles < 1 || n_ktiles < 1 || planes < 1) return 1;
  const double sms = num_sms > 0 ? num_sms : 1;
  // key tiles summed over the query tiles of one (batch, head)
  const double nq = n_qtiles, nk = n_ktiles;
  const double ksum = !causal ? nq * nk
                      : (nq <= nk ? nq * (nq + 1) / 2 : nk * (nk + 1) / 2 + (nq - nk) * nk);
  const double nbar = ksum / nq;
  const double tile = d <= 64 ? 0.5 : d <= 128 ? 1.0 : 2.0;  // relative key-tile time
  const double c = 2.6 / tile, c1 = 3.9 / tile;
  const double qtiles = static_cast<double>(planes) * n_qtiles;
  double best = causal ? qtiles * (nbar + c1) / sms + nbar
                       : std::ceil(qtiles / sms) * (nbar + c1);
  int pick = 1;
  for (int g = 2; g <= 4 && g <= n_qtiles; g *= 2) {
    const double ctas = static_cast<double>(planes) * std::ceil(nq / g);
    if (ctas < sms) break;
    const double cost = std::ceil(ctas / sms) * (g * nbar + c);
    if (cost < best) {
      best = cost;
      pick = g;
    }
  }
  return pick;
}

// Waves of items above which the blocked schedule replaces the persistent
// one.  Measured on GB300 (bf16, causal, d = 128): persistent ran 25% faster
// on b2h8n3001 (2.5 waves of query tiles) and 3% on b2h16n8192 (13.5 waves);
// blocked ran 4% faster on b8h32n8192 (108 waves) — the hardware hands out
// many CTAs as SMs free up, which evens out SMs that run at different speeds,
// where a fixed assignment waits for the slowest.
constexpr double kPersistentMaxWaves = 16.0;

// Schedule of the plain 16-bit forward (see fwd_item): *ctas CTAs of a 1-D
// grid, *group_heads planes per group (persistent), *block_items query
// tiles per CTA (blocked; 0 = persistent).  A test can force the persistent
// grid size
// (forced > 0), its group size (forced_group > 0) or the blocked schedule
// (forced_block > 0).  Other dtypes run one CTA per query tile (*ctas = 0).
void fwd_schedule(int dtype, int d, int causal, long long planes, int n_qtiles, int Nk,
                  int num_sms, int forced, int forced_group, int forced_block, int *ctas,
                  int *group_heads, int *block_items) {
  *ctas = 0;
  *group_heads = 1;
  *block_items = 0;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return;
  const long long items = planes * n_qtiles;
  const double sms = num_sms > 0 ? num_sms : 1;
  int block = forced_block;
  if (block <= 0 && forced <= 0 && forced_group <= 0 && items > kPersistentMaxWaves * sms)
    block = blocked_items(d, causal, planes, n_qtiles, (Nk + fa::BN - 1) / fa::BN, num_sms);
  if (block > 0) {
    const long long grid = planes * ((n_qtiles + block - 1) / block);
    if (grid <= 2147483647LL) {
      *ctas = static_cast<int>(grid);
      *block_items = block;
      return;
    }
  }
  long long c = forced > 0 ? forced : static_cast<long long>(sms);
  if (c > items) c = items;
  *ctas = static_cast<int>(c);
  const double kv = 2.0 * Nk * (d < 64 ? 64 : d) * static_cast<double>(elem_size(dtype));
  long long g = forced_group > 0 ? forced_group : static_cast<long long>(kL2GroupBytes / kv);
  if (g < 1) g = 1;
  if (g > planes) g = planes;
  *group_heads = static_cast<int>(g);
}

// The tensor-core forward instantiation for (dtype, d); the combination has
// been checked by validate().
//
// Head dim 32 runs on the d = 64 kernels zero-padded: the tensor maps over the
// 32-wide rows zero-fill columns 32..63 on load (so S and P V are unchanged)
// and clip them on store; d_io tells the kernel where its plain loads and
// stores stop.
//
// mklo: the staged fp32 path's map over K_lo (null otherwise; the kernels
// then get the K map in its place and never read it).
cudaError_t launch_tc_any(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const CUtensorMap &mo, const fa::TcParams &p_in, int B, int causal,
                          int d, int dtype, cudaStream_t s,
                          const CUtensorMap *mklo = nullptr) {
  fa::TcParams p = p_in;
  if (d == 32) {
    p.d_io = 32;
    d = 64;
  }
  const CUtensorMap &ml = mklo ? *mklo : mk;
  if (dtype == FA_DTYPE_F16)
    return d == 64    ? fa::launch_tc_f16_d64(mq, mk, mv, mo, ml, p, B, causal, s)
           : d == 128 ? fa::launch_tc_f16_d128(mq, mk, mv, mo, ml, p, B, causal, s)
                      : fa::launch_tc_f16_d256(mq, mk, mv, mo, ml, p, B, causal, s);
  if (dtype == FA_DTYPE_BF16)
    return d == 64    ? fa::launch_tc_bf16_d64(mq, mk, mv, mo, ml, p, B, causal, s)
           : d == 128 ? fa::launch_tc_bf16_d128(mq, mk, mv, mo, ml, p, B, causal, s)
                      : fa::launch_tc_bf16_d256(mq, mk, mv, mo, ml, p, B, causal, s);
  return d == 64 ? fa::launch_tc_f32_d64(mq, mk, mv, mo, ml, p, B, causal, s)
                 : fa::launch_tc_f32_d128(mq, mk, mv, mo, ml, p, B, causal, s);
}

// Extents of Q (= O) and LSE for the debug build's index checks: `rows`
// query rows of d elements.  A test can understate the LSE extent
// (fa_set_debug_lse_shrink) to make the checks fire without any access
// leaving the buffers.
void set_extents(fa::TcParams *p, long long rows, int d) {
  p->q_elems = rows * d;
  p->lse_elems = rows - g_dbg_lse_shrink.load();
}

// The tensor-core kernels take |scale| * log2(e) > 0 and apply a negative
// scale by negating Q inside the S = Q K^T product.  A zero scale becomes
// 1e-30: for scores below 1e20 in magnitude every exponent is then below
// 2^-40, so each exp2 rounds to exactly 1 and the weights are exactly uniform,
// as they are for scale 0.
void set_tc_scale(float scale, fa::TcParams *p) {
  const double a = scale == 0.f ? 1e-30 : std::fabs(static_cast<double>(scale));
  p->scale_log2 = static_cast<float>(a * 1.4426950408889634);
  p->scale_neg = scale < 0.f ? 1 : 0;
}

// The forward on device buffers once the arguments are validated: the SIMT
// kernel or the tensor-core kernel for (dtype, d), reporting bounded-wait
// give-ups into `status`.  Shared by fa_fwd and fa_fwd_noalloc, which differ
// only in where that word lives.
int fwd_enqueue(unsigned *status, const void *q, const void *k, const void *v, void *o,
                float *lse, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                int dtype, cudaStream_t s) {
  if (dtype == FA_DTYPE_F32_SIMT) {
    fa::SimtParams p;
    p.q = static_cast<const float *>(q);
    p.k = static_cast<const float *>(k);
    p.v = static_cast<const float *>(v);
    p.o = static_cast<float *>(o);
    p.lse = lse;
    p.status = status;
    p.B = B;
    p.H = H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.n_qtiles = ceil_div(Nq, fa::BM);
    p.scale = scale;
    p.causal = causal;
    p.num_sms = sm_count();
    return fa::launch_simt(p, B, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }

  int rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  CUtensorMap mq, mk, mv, mo;
  const int BH = B * H;  // <= 2^31 - 1 (validate)
  if ((rc = encode_map(&mq, q, dtype, BH, Nq, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mk, k, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mv, v, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mo, o, dtype, BH, Nq, d)) != FA_OK) return rc;

  fa::TcParams p;
  p.q = q;
  p.o = o;
  p.q_head_stride = static_cast<long long>(Nq) * d;
  p.q_row_stride = d;
  p.lse_head_stride = Nq;
  set_extents(&p, static_cast<long long>(B) * H * Nq, d);
  p.lse = lse;
  p.status = status;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qtiles = ceil_div(Nq, fa::BM);
  p.n_ktiles = ceil_div(Nk, fa::BN);
  set_tc_scale(scale, &p);
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.skip_v_load = g_skip_v_load.load();
  p.planes = BH;
  fwd_schedule(dtype, d, causal, BH, p.n_qtiles, Nk, sm_count(), g_force_ctas.load(),
               g_force_group.load(), g_force_block.load(), &p.ctas, &p.group_heads,
               &p.block_items);

  cudaError_t e = launch_tc_any(mq, mk, mv, mo, p, B, causal, d, dtype, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int Nq, int Nk, int d, float scale, int causal, int dtype, void *stream) {
  int rc = validate(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  return fwd_enqueue(status, q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype,
                     static_cast<cudaStream_t>(stream));
}

// fa_fwd_host's pipeline: per device, a stream for host->device copies, one
// for device->host copies and an event per chunk for each hand-over, made on
// first use and kept for the process (like the status word).  One call at a
// time per device uses them (the call is synchronous; a mutex serialises
// concurrent callers).
constexpr int kHostChunks = 8;
struct HostPipe {
  bool ready = false;
  std::mutex mu;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t loaded[kHostChunks] = {}, done[kHostChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe **pipe) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  HostPipe &hp = g_pipe[dev];
  std::lock_guard<std::mutex> lock(g_mu);
  if (!hp.ready) {
    if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int c = 0; c < kHostChunks; ++c)
      if (cudaEventCreateWithFlags(&hp.loaded[c], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.done[c], cudaEventDisableTiming) != cudaSuccess)
        return FA_ERR_CUDA;
    hp.ready = true;
  }
  *pipe = &hp;
  return FA_OK;
}

int fa_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d, int B, int H, int Nq,
                int Nk, int d, float scale, int causal, int dtype, void *stream) {
  if (!q_h || !k_h || !v_h || !o_h || !lse_h) return FA_ERR_INVALID_ARG;
  int rc = validate(q_d, k_d, v_d, o_d, lse_d, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  HostPipe *hp = nullptr;
  if ((rc = host_pipe(&hp)) != FA_OK) return rc;
  std::lock_guard<std::mutex> call_lock(hp->mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The (batch, head) planes are independent: chunk c's inputs go in on
  // hp->in, its forward runs on `stream` once they have landed, its outputs
  // come back on hp->out once it has finished, so the copies in, the
  // kernels and the copies out of different chunks overlap.
  const size_t es = elem_size(dtype);
  const size_t q_plane = static_cast<size_t>(Nq) * d * es, k_plane = static_cast<size_t>(Nk) * d * es;
  const size_t l_plane = static_cast<size_t>(Nq) * sizeof(float);
  const long long planes = static_cast<long long>(B) * H;
  // One chunk per 64 MB copied in (up to eight): small problems run as one
  // (there the launches and events of several would outweigh the overlap;
  // b2h4n1024d64 went from 19 to 8 TFLOP/s with eight).
  const size_t in_bytes = static_cast<size_t>(planes) * (q_plane + 2 * k_plane);
  size_t want = in_bytes / (size_t{64} << 20);
  if (want < 1) want = 1;
  if (want > static_cast<size_t>(kHostChunks)) want = kHostChunks;
  int nch = planes < static_cast<long long>(want) ? static_cast<int>(planes) : static_cast<int>(want);
  // A chunk runs as a problem of its planes with one head each, and the grid
  // takes at most 65535 of them: beyond that the whole problem runs as one.
  if ((planes + nch - 1) / nch > 65535) nch = 1;
  // the inputs must not be overwritten while an earlier call's work on
  // `stream` may still read them
  if (cudaEventRecord(hp->done[0], s) != cudaSuccess ||
      cudaStreamWaitEvent(hp->in, hp->done[0], 0) != cudaSuccess)
    return FA_ERR_CUDA;
  auto ptr = [](const void *base, size_t off) {
    return static_cast<void *>(static_cast<char *>(const_cast<void *>(base)) + off);
  };
  int first_rc = FA_OK;
  for (int c = 0; c < nch && first_rc == FA_OK; ++c) {
    const long long p0 = planes * c / nch, p1 = planes * (c + 1) / nch;
    const long long np = p1 - p0;
    if (np == 0) continue;
    if (cudaMemcpyAsync(ptr(q_d, p0 * q_plane), ptr(q_h, p0 * q_plane), np * q_plane,
                        cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(ptr(k_d, p0 * k_plane), ptr(k_h, p0 * k_plane), np * k_plane,
                        cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(ptr(v_d, p0 * k_plane), ptr(v_h, p0 * k_plane), np * k_plane,
                        cudaMemcpyHostToDevice, hp->in) != cudaSuccess ||
        cudaEventRecord(hp->loaded[c], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(s, hp->loaded[c], 0) != cudaSuccess) {
      first_rc = FA_ERR_CUDA;
      break;
    }
    // the chunk as a problem of np planes of one head each (one chunk: the
    // problem as given)
    const int cb = nch == 1 ? B : static_cast<int>(np), ch = nch == 1 ? H : 1;
    const int rc_c = fa_fwd(ptr(q_d, p0 * q_plane), ptr(k_d, p0 * k_plane),
                            ptr(v_d, p0 * k_plane), ptr(o_d, p0 * q_plane),
                            static_cast<float *>(ptr(lse_d, p0 * l_plane)), cb, ch, Nq, Nk, d,
                            scale, causal, dtype, stream);
    if (rc_c != FA_OK) {
      first_rc = rc_c;
      break;
    }
    if (cudaEventRecord(hp->done[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->done[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(ptr(o_h, p0 * q_plane), ptr(o_d, p0 * q_plane), np * q_plane,
                        cudaMemcpyDeviceToHost, hp->out) != cudaSuccess ||
        cudaMemcpyAsync(ptr(lse_h, p0 * l_plane), ptr(lse_d, p0 * l_plane), np * l_plane,
                        cudaMemcpyDeviceToHost, hp->out) != cudaSuccess) {
      first_rc = FA_ERR_CUDA;
      break;
    }
  }
  // Everything enqueued has finished before the call returns (also after a
  // failure, so no copy still runs into the caller's buffers).
  const bool synced = cudaStreamSynchronize(hp->in) == cudaSuccess &&
                      cudaStreamSynchronize(s) == cudaSuccess &&
                      cudaStreamSynchronize(hp->out) == cudaSuccess;
  if (first_rc != FA_OK) return first_rc;
  return synced ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_status(void *stream, int *device_status) {
  if (device_status) *device_status = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  unsigned *ptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ptr = g_status[dev];
  }
  if (ptr == nullptr) return FA_OK;  // nothing has run on this device
  unsigned word = 0;
  if (cudaMemcpy(&word, ptr, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word != 0 && cudaMemset(ptr, 0, sizeof word) != cudaSuccess) return FA_ERR_CUDA;
  if (device_status) *device_status = static_cast<int>(word);
  return word ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_version(void) { return FA_VERSION; }

int fa_set_test_hooks(int skip_v_load, unsigned long long wait_limit_ns) {
  g_skip_v_load.store(skip_v_load ? 1 : 0);
  g_wait_limit_ns.store(wait_limit_ns);
  return FA_OK;
}

int fa_fwd_schedule(int B, int H, int Nq, int Nk, int d, int causal, int dtype, int num_sms,
                    int *ctas, int *group_heads, int *block_items) {
  if (!ctas || !group_heads || !block_items) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1 || num_sms < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 2147483647LL) return FA_ERR_INVALID_ARG;
  fwd_schedule(dtype, d, causal, static_cast<long long>(B) * H, ceil_div(Nq, fa::BM), Nk, num_sms,
               g_force_ctas.load(), g_force_group.load(), g_force_block.load(), ctas,
               group_heads, block_items);
  return FA_OK;
}

int fa_fwd_schedule_covers(int planes, int n, int ctas, int group_heads, int block_items) {
  if (planes < 1 || n < 1 || ctas < 1 || group_heads < 1 || block_items < 0) return 0;
  const long long items = static_cast<long long>(planes) * n;
  if (items > (1LL << 24)) return 0;
  if (block_items == 0 && ctas > items) return 0;
  if (block_items > 0 &&
      ctas != static_cast<long long>(planes) * ((n + block_items - 1) / block_items))
    return 0;
  std::vector<unsigned char> seen(static_cast<size_t>(items), 0);
  for (int c = 0; c < ctas; ++c) {
    for (int k = 0;; ++k) {
      int plane = -1;
      const int t = fa::fwd_item(k, c, ctas, planes, n, group_heads, block_items, &plane);
      if (t < 0) break;
      if (t >= n || plane < 0 || plane >= planes) return 0;
      unsigned char &v = seen[static_cast<size_t>(plane) * n + t];
      if (v) return 0;
      v = 1;
    }
  }
  for (unsigned char v : seen)
    if (!v) return 0;
  return 1;
}

int fa_debug_build(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

int fa_set_debug_lse_shrink(long long elems) {
#ifdef FA_DEBUG
  if (elems < 0) return FA_ERR_INVALID_ARG;
  g_dbg_lse_shrink.store(elems);
  return FA_OK;
#else
  (void)elems;
  return FA_ERR_UNSUPPORTED;
#endif
}

int fa_set_fwd_schedule(int ctas, int group_heads, int block_items) {
  if (ctas < 0 || group_heads < 0 || block_items < 0) return FA_ERR_INVALID_ARG;
  g_force_ctas.store(ctas);
  g_force_group.store(group_heads);
  g_force_block.store(block_items);
  return FA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// No-allocation variant.
//
// fa_fwd keeps its per-device status word in memory it obtains with
// cudaMalloc on the first call.  Some callers cannot let a library do that: a
// serving process that reserves all of the GPU's memory for its own pool at
// start-up (a cudaMalloc from inside a call then fails, or eats into memory
// the pool has promised elsewhere), a latency-critical loop where the implicit
// device-wide synchronisation of cudaMalloc would stall other streams, or a
// framework whose memory manager must account for every device allocation.
// fa_fwd_noalloc gives them the same forward with the status word kept in a
// fixed array that is part of the library's device image instead.
// ---------------------------------------------------------------------------
namespace {

// Scratch of the no-allocation path: word 0 is the status word the kernels OR
// their give-up bits into; the rest is padding to the alignment.  It is part
// of the library's device image, so every GPU that loads the library holds
// these 256 bytes until the process exits.  All calls share it.
constexpr size_t kNoallocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

unsigned *g_noalloc_status[kMaxDevices] = {};  // device address of word 0, per device

// sm_103 check and the scratch's device address for the current device; the
// address is looked up once per device, with that device current.
int noalloc_setup(unsigned **status) {
  int rc, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if ((rc = check_sm103(dev)) != FA_OK) return rc;
  if (g_noalloc_status[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_CUDA;
    g_noalloc_status[dev] = static_cast<unsigned *>(ptr);
  }
  *status = g_noalloc_status[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int Nq, int Nk, int d, float scale, int causal,
                              int dtype, void *stream, int *device_status) {
  if (device_status) *device_status = 0;
  int rc = validate(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  // Scratch this call needs: one status word, whatever the problem size.
  const size_t need = sizeof(unsigned);
  if (need > kNoallocScratchBytes) return FA_ERR_UNSUPPORTED;
  unsigned *status = nullptr;
  if ((rc = noalloc_setup(&status)) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start
  // at zero for this call.
  if (cudaMemsetAsync(status, 0, need, s) != cudaSuccess) return FA_ERR_CUDA;
  if ((rc = fwd_enqueue(status, q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, s)) !=
      FA_OK)
    return rc;
  if (device_status == nullptr) return FA_OK;
  // Synchronous form: wait for the kernel and report its status word.
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, status, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FA_ERR_CUDA;
  *device_status = static_cast<int>(word);
  return word ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

// ---------------------------------------------------------------------------
// Split over the key range.
// ---------------------------------------------------------------------------
namespace {

constexpr int kMaxSplits = 64;

size_t splitkv_ws_bytes(int B, int H, int Nq, int d, int nsp) {
  const size_t rows = static_cast<size_t>(nsp) * B * H * Nq;
  const size_t o_bytes = (rows * d * sizeof(float) + 255) & ~static_cast<size_t>(255);
  const size_t l_bytes = (rows * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return o_bytes + l_bytes;
}

int sm_count() {
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count[dev] = c;
  }
  return count[dev];
}

}  // namespace

extern "C" unsigned long long fa_fwd_splitkv_workspace(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_ws_bytes(B, H, Nq, d, num_splits);
}

extern "C" int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int Nq, int Nk, int d, float scale, int causal,
                              int dtype, int num_splits, void *workspace,
                              unsigned long long workspace_bytes, void *stream) {
  int rc = validate(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32_SIMT) return FA_ERR_UNSUPPORTED;
  const int n_qtiles = ceil_div(Nq, fa::BM), n_ktiles = ceil_div(Nk, fa::BN);
  if (num_splits > 0) {
    // The workspace is checked before anything touches the device.
    const size_t need = splitkv_ws_bytes(B, H, Nq, d, num_splits);
    if (num_splits > 1 &&
        (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
         workspace_bytes < need))
      return FA_ERR_INVALID_ARG;
  }
  int nsp = num_splits;
  if (nsp == 0) {
    // One wave: about one CTA per SM (a CTA holds a whole SM's tensor
    // memory, so a second wave would run after the first), at least one key
    // tile per chunk.
    const int sms = sm_count();
    if (sms == 0) return FA_ERR_CUDA;
    const long long ctas = static_cast<long long>(n_qtiles) * B * H;
    nsp = static_cast<int>(sms / ctas);
    nsp = nsp < 1 ? 1 : (nsp > n_ktiles ? n_ktiles : nsp);
    if (nsp > kMaxSplits) nsp = kMaxSplits;
    while (nsp > 1 && (workspace == nullptr ||
                       reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
                       workspace_bytes < splitkv_ws_bytes(B, H, Nq, d, nsp)))
      --nsp;  // the largest split count the workspace holds
  }
  if (nsp <= 1) return fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream);
  const size_t need = splitkv_ws_bytes(B, H, Nq, d, nsp);
  const size_t o_part = need - ((static_cast<size_t>(nsp) * B * H * Nq * sizeof(float) + 255) &
                                ~static_cast<size_t>(255));
  float *ws_o = static_cast<float *>(workspace);
  float *ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_part);
  if (overlap(workspace, need, q, static_cast<size_t>(B) * H * Nq * d * elem_size(dtype)) ||
      overlap(workspace, need, k, static_cast<size_t>(B) * H * Nk * d * elem_size(dtype)) ||
      overlap(workspace, need, v, static_cast<size_t>(B) * H * Nk * d * elem_size(dtype)) ||
      overlap(workspace, need, o, static_cast<size_t>(B) * H * Nq * d * elem_size(dtype)) ||
      overlap(workspace, need, lse, static_cast<size_t>(B) * H * Nq * sizeof(float)))
    return FA_ERR_INVALID_ARG;

  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap mq, mk, mv, mo;
  const int BH = B * H;
  if ((rc = encode_map(&mq, q, dtype, BH, Nq, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mk, k, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mv, v, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mo, o, dtype, BH, Nq, d)) != FA_OK) return rc;
  fa::TcParams p;
  p.q = q;
  p.o = o;
  p.q_head_stride = static_cast<long long>(Nq) * d;
  p.q_row_stride = d;
  p.lse_head_stride = Nq;
  set_extents(&p, static_cast<long long>(B) * H * Nq, d);
  p.lse = lse;
  p.status = status;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qtiles = n_qtiles;
  p.n_ktiles = n_ktiles;
  set_tc_scale(scale, &p);
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.skip_v_load = g_skip_v_load.load();
  p.n_splits = nsp;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  cudaError_t e = launch_tc_any(mq, mk, mv, mo, p, B, causal, d, dtype, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  e = fa::launch_splitkv_combine(ws_o, ws_lse, o, lse, BH, Nq, d, n_ktiles, nsp, causal, dtype,
                                 status, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Variable-length batches.
// ---------------------------------------------------------------------------
namespace {

// 3-D view {d, total rows, H} of a token-major [total, H, d] tensor: rows of
// one head are H*d elements apart, heads d apart.  Boxes as encode_map.
int encode_map_tokens(CUtensorMap *map, const void *base, int dtype, int total, int H, int d) {
  const CUtensorMapDataType dt = dtype == FA_DTYPE_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == FA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t es = elem_size(dtype);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(total),
                        static_cast<cuuint64_t>(H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * d * es, static_cast<cuuint64_t>(d) * es};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(fa::BM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                             const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                             int total_q, int total_k, int max_seqlen_q, int d, float scale,
                             int causal, int dtype, void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cu_seqlens_q) % 4 || reinterpret_cast<uintptr_t>(cu_seqlens_k) % 4)
    return FA_ERR_INVALID_ARG;
  if (max_seqlen_q < 1 || max_seqlen_q > total_q) return FA_ERR_INVALID_ARG;
  // The tensors as one [1, H, total, d]-sized problem for the shared checks
  // (pointers, alignment, sizes, overlaps, supported dtype and d).
  int rc = validate(q, k, v, o, lse, 1, H, total_q, total_k, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  if (B < 1 || B > 65535) return FA_ERR_INVALID_ARG;
  if (dtype == FA_DTYPE_F32_SIMT) return FA_ERR_UNSUPPORTED;
  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap mq, mk, mv, mo;
  if ((rc = encode_map_tokens(&mq, q, dtype, total_q, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mk, k, dtype, total_k, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mv, v, dtype, total_k, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mo, o, dtype, total_q, H, d)) != FA_OK) return rc;
  fa::TcParams p;
  p.q = q;
  p.o = o;
  p.lse = lse;
  p.status = status;
  p.H = H;
  p.Nq = max_seqlen_q;
  p.Nk = total_k;
  p.n_qtiles = ceil_div(max_seqlen_q, fa::BM);  // grid: the longest sequence
  p.n_ktiles = ceil_div(total_k, fa::BN);
  set_tc_scale(scale, &p);
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.skip_v_load = g_skip_v_load.load();
  p.q_head_stride = d;
  p.q_row_stride = static_cast<long long>(H) * d;
  p.lse_head_stride = total_q;
  set_extents(&p, static_cast<long long>(H) * total_q, d);
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = total_q;
  p.total_k = total_k;
  cudaError_t e = launch_tc_any(mq, mk, mv, mo, p, B, causal, d, dtype, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Backward.
// ---------------------------------------------------------------------------
namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Row length of the fp32 dQ accumulator: the gradient kernel's head dim
// (d = 32 runs on the d = 64 kernel).
size_t bwd_acc_dim(int d) { return d < 64 ? 64 : static_cast<size_t>(d); }

// Workspace parts: dq_acc [B*H][Nq][max(d, 64)] fp32, then lse2 and dd
// [B*H][Nq_pad].
void bwd_ws_parts(int B, int H, int Nq, int d, size_t *acc, size_t *row) {
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t nq_pad = static_cast<size_t>(ceil_div(Nq, fa::BM)) * fa::BM;
  *acc = round256(bh * Nq * bwd_acc_dim(d) * sizeof(float));
  *row = round256(bh * nq_pad * sizeof(float));
}

}  // namespace

extern "C" unsigned long long fa_bwd_workspace(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1) return 0;
  size_t acc, row;
  bwd_ws_parts(B, H, Nq, d, &acc, &row);
  return acc + 2 * row;
}

extern "C" int fa_bwd(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                      int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
                      void *workspace, unsigned long long workspace_bytes, void *stream) {
  // The forward's checks cover q, k, v, o, lse, the sizes, scale and dtype.
  int rc = validate(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  if (!dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  for (const void *ptr : {dout, static_cast<const void *>(dq), static_cast<const void *>(dk),
                          static_cast<const void *>(dv)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return FA_ERR_INVALID_ARG;
  size_t acc, row;
  bwd_ws_parts(B, H, Nq, d, &acc, &row);
  const size_t need = acc + 2 * row;
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t qn = static_cast<size_t>(B) * H * Nq * d * es;
  const size_t kn = static_cast<size_t>(B) * H * Nk * d * es;
  const size_t ln = static_cast<size_t>(B) * H * Nq * sizeof(float);
  // Outputs and workspace must not overlap each other or any input.
  const struct { const void *p; size_t n; } in[] = {{q, qn}, {k, kn}, {v, kn}, {o, qn},
                                                    {lse, ln}, {dout, qn}};
  const struct { const void *p; size_t n; } out[] = {{dq, qn}, {dk, kn}, {dv, kn},
                                                     {workspace, need}};
  for (int a = 0; a < 4; ++a) {
    for (const auto &x : in)
      if (overlap(out[a].p, out[a].n, x.p, x.n)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlap(out[a].p, out[a].n, out[b].p, out[b].n)) return FA_ERR_INVALID_ARG;
  }
  if (dtype == FA_DTYPE_F32 || dtype == FA_DTYPE_F32_SIMT) {
    // fp32: the CUDA-core backward (head dim up to 128); the workspace
    // holds D per query row.
    if (d > 128) return FA_ERR_UNSUPPORTED;
    unsigned *status = nullptr;
    if ((rc = device_setup(&status)) != FA_OK) return rc;
    const cudaError_t e = fa::launch_bwd_simt(
        static_cast<const float *>(q), static_cast<const float *>(k),
        static_cast<const float *>(v), static_cast<const float *>(o), lse,
        static_cast<const float *>(dout), static_cast<float *>(dq), static_cast<float *>(dk),
        static_cast<float *>(dv), static_cast<float *>(workspace), B, H, Nq, Nk, d, scale, causal,
        status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  // d = 32 runs zero-padded on the d = 64 kernel; dK, dV of d = 256 do not
  // fit in tensor memory.
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;

  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = encode_map(&mq, q, dtype, BH, Nq, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mk, k, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mv, v, dtype, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mdo, dout, dtype, BH, Nq, d)) != FA_OK) return rc;

  fa::BwdParams p;
  p.dq_acc = static_cast<float *>(workspace);
  float *lse2 = reinterpret_cast<float *>(static_cast<char *>(workspace) + acc);
  float *dd = reinterpret_cast<float *>(static_cast<char *>(workspace) + acc + row);
  p.lse2 = lse2;
  p.dd = dd;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qtiles = ceil_div(Nq, fa::BM);
  p.n_ktiles = ceil_div(Nk, fa::BN);
  p.Nq_pad = p.n_qtiles * fa::BM;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.d_io = d == 32 ? 32 : 0;
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.dq_elems = static_cast<long long>(BH) * Nq * static_cast<long long>(bwd_acc_dim(d));
  p.row_elems = static_cast<long long>(BH) * p.Nq_pad;
  p.kv_elems = static_cast<long long>(BH) * Nk * d;
  const int half = dtype == FA_DTYPE_F16 ? 1 : 0;

  cudaError_t e = fa::launch_bwd_prep(o, dout, lse, lse2, dd, p.dq_acc, BH, Nq, p.Nq_pad, d,
                                      half, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (half)
    e = (d <= 64) ? fa::launch_bwd_f16_d64(mq, mk, mv, mdo, p, B, causal, s)
                  : fa::launch_bwd_f16_d128(mq, mk, mv, mdo, p, B, causal, s);
  else
    e = (d <= 64) ? fa::launch_bwd_bf16_d64(mq, mk, mv, mdo, p, B, causal, s)
                  : fa::launch_bwd_bf16_d128(mq, mk, mv, mdo, p, B, causal, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  e = fa::launch_bwd_convert(p.dq_acc, dq, static_cast<long long>(BH) * Nq, d, H, 0, half, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Forward with a staging workspace (fp32: operands converted once per call).
// ---------------------------------------------------------------------------
namespace {

int nk_pad128(int Nk) { return ceil_div(Nk, fa::BN) * fa::BN; }

// Workspace parts for fp32: K_hi = tf32(K) [B*H][Nk][d], K_lo =
// tf32(K - K_hi) [B*H][Nk][d] (each part kr bytes), then V^T
// [B*H][d][Nk padded to 128].
void staged_parts(int B, int H, int Nk, int d, size_t *kr, size_t *vt) {
  const size_t bh = static_cast<size_t>(B) * H;
  *kr = round256(bh * Nk * d * sizeof(__nv_bfloat16));  // one bf16 half of the split K
  *vt = round256(bh * d * static_cast<size_t>(nk_pad128(Nk)) * sizeof(float));
}

// 3-D view {Nk_pad, d, B*H} of the staged V^T, boxes of 32 keys (128 bytes)
// x dk rows (the kernel's head dim; rows past d read as zeros).
int encode_map_vt(CUtensorMap *map, void *base, int BH, int nk_pad, int d, int dk) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(nk_pad), static_cast<cuuint64_t>(d),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(nk_pad) * 4,
                           static_cast<cuuint64_t>(nk_pad) * static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[3] = {32, static_cast<cuuint32_t>(dk), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" unsigned long long fa_fwd_staged_workspace(int B, int H, int Nk, int d, int dtype) {
  if (B < 1 || H < 1 || Nk < 1 || d < 1) return 0;
  if (dtype != FA_DTYPE_F32) return 0;  // only the fp32 path stages operands
  size_t kr, vt;
  staged_parts(B, H, Nk, d, &kr, &vt);
  return 2 * kr + vt;
}

extern "C" int fa_fwd_staged(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int Nq, int Nk, int d, float scale, int causal,
                             int dtype, void *workspace, unsigned long long workspace_bytes,
                             void *stream) {
  int rc = validate(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  if (dtype != FA_DTYPE_F32)  // nothing to stage
    return fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, stream);
  size_t kr_bytes, vt_bytes;
  staged_parts(B, H, Nk, d, &kr_bytes, &vt_bytes);
  const size_t need = 2 * kr_bytes + vt_bytes;
  if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
      workspace_bytes < need)
    return FA_ERR_INVALID_ARG;
  const size_t qn = static_cast<size_t>(B) * H * Nq * d * 4;
  const size_t kn = static_cast<size_t>(B) * H * Nk * d * 4;
  const size_t ln = static_cast<size_t>(B) * H * Nq * sizeof(float);
  if (overlap(workspace, need, q, qn) || overlap(workspace, need, k, kn) ||
      overlap(workspace, need, v, kn) || overlap(workspace, need, o, qn) ||
      overlap(workspace, need, lse, ln))
    return FA_ERR_INVALID_ARG;

  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H, nkp = nk_pad128(Nk);
  auto *kr = static_cast<__nv_bfloat16 *>(workspace);
  auto *kl = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(workspace) + kr_bytes);
  float *vt = reinterpret_cast<float *>(static_cast<char *>(workspace) + 2 * kr_bytes);
  if (fa::launch_stage_f32(static_cast<const float *>(k), static_cast<const float *>(v), kr, kl,
                           vt, BH, Nk, nkp, d, s) != cudaSuccess)
    return FA_ERR_CUDA;

  CUtensorMap mq, mk, mv, mo, mkl;
  if ((rc = encode_map(&mq, q, dtype, BH, Nq, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mk, kr, FA_DTYPE_BF16, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map(&mkl, kl, FA_DTYPE_BF16, BH, Nk, d)) != FA_OK) return rc;
  if ((rc = encode_map_vt(&mv, vt, BH, nkp, d, d <= 64 ? 64 : 128)) != FA_OK) return rc;
  if ((rc = encode_map(&mo, o, dtype, BH, Nq, d)) != FA_OK) return rc;
  fa::TcParams p;
  p.q = q;
  p.o = o;
  p.q_head_stride = static_cast<long long>(Nq) * d;
  p.q_row_stride = d;
  p.lse_head_stride = Nq;
  set_extents(&p, static_cast<long long>(B) * H * Nq, d);
  p.lse = lse;
  p.status = status;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qtiles = ceil_div(Nq, fa::BM);
  p.n_ktiles = ceil_div(Nk, fa::BN);
  set_tc_scale(scale, &p);
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.skip_v_load = g_skip_v_load.load();
  p.kv_staged = 1;
  if (d == 32) {
    p.d_io = 32;
    d = 64;
  }
  cudaError_t e = d == 64 ? fa::launch_tc_f32s_d64(mq, mk, mv, mo, mkl, p, B, causal, s)
                          : fa::launch_tc_f32s_d128(mq, mk, mv, mo, mkl, p, B, causal, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Backward over variable-length batches.
// ---------------------------------------------------------------------------
namespace {

// Workspace parts: dq_acc [H][total_q][max(d, 64)] fp32, then lse2 and dd
// [H][B][Nq_pad].
void bwd_varlen_parts(int B, int H, int total_q, int max_q, int d, size_t *acc, size_t *row) {
  const size_t pad = static_cast<size_t>(ceil_div(max_q, fa::BM)) * fa::BM;
  *acc = round256(static_cast<size_t>(total_q) * H * bwd_acc_dim(d) * sizeof(float));
  *row = round256(static_cast<size_t>(H) * B * pad * sizeof(float));
}

}  // namespace

extern "C" unsigned long long fa_bwd_varlen_workspace(int B, int H, int total_q, int max_seqlen_q,
                                                      int d) {
  if (B < 1 || H < 1 || total_q < 1 || max_seqlen_q < 1 || d < 1) return 0;
  size_t acc, row;
  bwd_varlen_parts(B, H, total_q, max_seqlen_q, d, &acc, &row);
  return acc + 2 * row;
}

extern "C" int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                             float scale, int causal, int dtype, void *workspace,
                             unsigned long long workspace_bytes, void *stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cu_seqlens_q) % 4 || reinterpret_cast<uintptr_t>(cu_seqlens_k) % 4)
    return FA_ERR_INVALID_ARG;
  if (max_seqlen_q < 1 || max_seqlen_q > total_q || max_seqlen_k < 1 || max_seqlen_k > total_k)
    return FA_ERR_INVALID_ARG;
  // The tensors as one [1, H, total, d]-sized problem for the shared checks.
  int rc = validate(q, k, v, o, lse, 1, H, total_q, total_k, d, scale, causal, dtype);
  if (rc != FA_OK) return rc;
  if (B < 1 || B > 65535) return FA_ERR_INVALID_ARG;
  if (!dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  for (const void *ptr : {dout, static_cast<const void *>(dq), static_cast<const void *>(dk),
                          static_cast<const void *>(dv)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return FA_ERR_INVALID_ARG;
  size_t acc, row;
  bwd_varlen_parts(B, H, total_q, max_seqlen_q, d, &acc, &row);
  const size_t need = acc + 2 * row;
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const size_t es = elem_size(dtype);
  const size_t qn = static_cast<size_t>(total_q) * H * d * es;
  const size_t kn = static_cast<size_t>(total_k) * H * d * es;
  const size_t ln = static_cast<size_t>(H) * total_q * sizeof(float);
  const struct { const void *p; size_t n; } in[] = {{q, qn}, {k, kn}, {v, kn}, {o, qn},
                                                    {lse, ln}, {dout, qn}};
  const struct { const void *p; size_t n; } out[] = {{dq, qn}, {dk, kn}, {dv, kn},
                                                     {workspace, need}};
  for (int a = 0; a < 4; ++a) {
    for (const auto &x : in)
      if (overlap(out[a].p, out[a].n, x.p, x.n)) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlap(out[a].p, out[a].n, out[b].p, out[b].n)) return FA_ERR_INVALID_ARG;
  }
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F16) return FA_ERR_UNSUPPORTED;
  if (d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;

  unsigned *status = nullptr;
  if ((rc = device_setup(&status)) != FA_OK) return rc;
  if ((rc = get_encoder()) != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = encode_map_tokens(&mq, q, dtype, total_q, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mk, k, dtype, total_k, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mv, v, dtype, total_k, H, d)) != FA_OK) return rc;
  if ((rc = encode_map_tokens(&mdo, dout, dtype, total_q, H, d)) != FA_OK) return rc;

  fa::BwdParams p;
  p.dq_acc = static_cast<float *>(workspace);
  float *lse2 = reinterpret_cast<float *>(static_cast<char *>(workspace) + acc);
  float *dd = reinterpret_cast<float *>(static_cast<char *>(workspace) + acc + row);
  p.lse2 = lse2;
  p.dd = dd;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.H = H;
  p.Nq = max_seqlen_q;
  p.Nk = max_seqlen_k;
  p.n_qtiles = ceil_div(max_seqlen_q, fa::BM);
  p.n_ktiles = ceil_div(max_seqlen_k, fa::BN);  // the grid covers the longest sequence
  p.Nq_pad = p.n_qtiles * fa::BM;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitLimitNs;
  p.d_io = d == 32 ? 32 : 0;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = total_q;
  p.total_k = total_k;
  p.dq_elems = static_cast<long long>(total_q) * H * static_cast<long long>(bwd_acc_dim(d));
  p.row_elems = static_cast<long long>(H) * B * p.Nq_pad;
  p.kv_elems = static_cast<long long>(total_k) * H * d;
  const int half = dtype == FA_DTYPE_F16 ? 1 : 0;

  cudaError_t e = fa::launch_bwd_prep_varlen(o, dout, lse, lse2, dd, p.dq_acc, cu_seqlens_q, B, H,
                                             total_q, p.Nq_pad, d, half, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (half)
    e = (d <= 64) ? fa::launch_bwd_f16_d64(mq, mk, mv, mdo, p, B, causal, s)
                  : fa::launch_bwd_f16_d128(mq, mk, mv, mdo, p, B, causal, s);
  else
    e = (d <= 64) ? fa::launch_bwd_bf16_d64(mq, mk, mv, mdo, p, B, causal, s)
                  : fa::launch_bwd_bf16_d128(mq, mk, mv, mdo, p, B, causal, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  e = fa::launch_bwd_convert(p.dq_acc, dq, static_cast<long long>(total_q) * H, d, H, total_q, half,
                             s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
