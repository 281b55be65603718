// fa_internal.h — declarations shared by the host API and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fa {

// The dynamic shared-memory opt-in of a kernel, set once per device: `done`
// keeps one bit per device (devices past 63 set it on every launch).  Saves a
// runtime call on every launch of a small problem.
template <typename Kernel>
cudaError_t smem_attr_once(Kernel kern, int bytes, std::atomic<unsigned long long> *done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
  if (bit != 0 && (done->load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done->fetch_or(bit, std::memory_order_release);
  return e;
}

// Tile shape of the tensor-core kernels: a query tile is BM rows of one
// (batch, head); the keys stream in tiles of BN.
constexpr int BM = 128;
constexpr int BN = 128;

// Status-word bits (see fa_fwd_status in fa.h).
constexpr unsigned kStatusProducer = 1u;
constexpr unsigned kStatusMma = 2u;
constexpr unsigned kStatusSoftmax = 4u;
constexpr unsigned kStatusInjected = 8u;
constexpr unsigned kStatusSmemLayout = 16u;  // shared memory base not aligned as needed
constexpr unsigned kStatusBounds = 32u;      // debug build: an index check failed

// Index checks of the debug build (compiled with FA_DEBUG): every plain
// global load and store of the kernels (those not made by TMA, whose tensor
// maps bound them already) first checks that elements [first, first+count)
// lie inside the buffer's `extent` elements; a failed check ORs
// kStatusBounds into the status word and the access is skipped, so a wrong
// index shows up in fa_fwd_status instead of faulting the GPU.  The release
// build compiles the checks away.
#ifdef FA_DEBUG
__device__ __forceinline__ bool dbg_in(unsigned *status, long long first, long long count,
                                       long long extent) {
  if (first >= 0 && count >= 0 && first + count <= extent) return true;
  atomicOr(status, kStatusBounds);
  return false;
}
#define FA_IN(status, first, count, extent)                                              \
  ::fa::dbg_in((status), static_cast<long long>(first), static_cast<long long>(count), \
               static_cast<long long>(extent))
#else
#define FA_IN(status, first, count, extent) true
#endif

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s

struct TcParams {
  const void *q;                  // [B*H*Nq*d], read row by row when Q goes to TMEM
  void *o;                        // output, written row by row for variable lengths
  float *lse;                     // [B*H*Nq]
  unsigned *status;               // per-device status word
  int H, Nq, Nk;
  int n_qtiles, n_ktiles;         // ceil(Nq/BM), ceil(Nk/BN)
  float scale_log2;               // |scale| * log2(e) > 0
  int scale_neg;                  // scale < 0: S is computed as (-Q) K^T
  unsigned long long wait_limit_ns;
  int skip_v_load;                // test hook
  // Split over the key range (1 = off): CTA x covers query tile x / n_splits
  // and chunk x % n_splits of that tile's key tiles, writing O/l (fp32) and
  // LSE of its chunk to ws_o [n_splits][B*H][Nq][d] and ws_lse [n_splits][B*H][Nq].
  int n_splits = 1;
  float *ws_o = nullptr;
  float *ws_lse = nullptr;
  // Element strides of Q and O (and of LSE) for the head coordinate and the
  // row: [B,H,N,d] uses (Nq*d, d) and Nq with the head coordinate b*H+h; the
  // variable-length layout [total, H, d] uses (d, H*d) and total_q with h.
  long long q_head_stride = 0, q_row_stride = 0, lse_head_stride = 0;
  // Variable-length batches: device cu_seqlens (B+1 entries each), or null.
  // Sequence b covers rows [cu_q[b], cu_q[b+1]) of Q/O and [cu_k[b], cu_k[b+1])
  // of K/V; total_q and total_k bound every row index (defends against bad
  // offsets).
  const int *cu_q = nullptr;
  const int *cu_k = nullptr;
  int total_q = 0, total_k = 0;
  // Head dim of the tensors when narrower than the kernel's D (0 = D): the
  // kernel runs zero-padded to D.
  int d_io = 0;
  // Elements of Q (= of O) and of LSE, for the debug build's index checks.
  long long q_elems = 0, lse_elems = 0;
  // fp32 path: K already split into K_hi (tm_k) and K_lo (tm_klo), and tm_v
  // a map over a tf32 V^T ([B*H][d][Nk padded to 128], boxes of 32 keys x D
  // rows).
  int kv_staged = 0;
  // Schedule of the plain problems of the 16-bit types (ctas > 0): a 1-D
  // grid of `ctas` CTAs, each running the query tiles ("items") fwd_item()
  // assigns it; planes = B*H; group_heads and block_items as in
  // fwd_item().  ctas = 0: one CTA per (query tile, head, batch) on a 3-D
  // grid.
  int ctas = 0;
  int planes = 0;
  int group_heads = 1;
  int block_items = 0;
};

// Item k of CTA c of a grid of P CTAs, for planes of n items (query tiles)
// each: returns the item's index within its
// plane and sets *plane (the (batch, head) index b*H + h), or returns -1
// when the CTA has no k-th item.  Item n-1 is the heaviest under causal
// masking (the most key tiles), item 0 the lightest.  Two schedules:
//
// block_items = 0, persistent (P is about one CTA per SM): the planes in
// groups of group_heads (a group's K and V are sized to stay in L2 while its
// items run); within a group, item n-1 of every plane, then n-2, and so on
// (heaviest first); dealt in rounds of P, alternately to CTAs 0..P-1 and
// P-1..0, so the heaviest and lightest items of successive rounds pair up
// and every CTA gets about the same work.  Suits grids of a few waves, where
// the last wave's imbalance would otherwise cost most.
//
// block_items = G >= 1, blocked (P = planes * ceil(n / G)): CTA c takes G
// consecutive positions of its plane's zigzag order (heaviest, lightest,
// next heaviest, ...), so with an even G every causal CTA has the same
// work; with G = 1 the CTAs of a plane go heaviest first.  CTAs of one plane
// are adjacent, and the hardware hands CTAs to SMs as they free up, which
// balances many waves better than any fixed assignment.
//
// Either way every item 0 .. planes*n-1 goes to exactly one (CTA, k).
__host__ __device__ inline int fwd_item(int k, int c, int P, int planes, int n, int group_heads,
                                        int block_items, int *plane) {
  if (block_items > 0) {
    const int nb = (n + block_items - 1) / block_items;  // CTAs per plane
    if (k >= block_items) return -1;
    *plane = c / nb;
    const int x = c - *plane * nb;
    if (block_items == 1) return n - 1 - x;
    const int zi = block_items * x + k;
    if (zi >= n) return -1;
    const int qi = (zi & 1) ? n - 1 - (zi >> 1) : (zi >> 1);
    return n - 1 - qi;
  }
  const long long i = static_cast<long long>(k) * P + ((k & 1) ? P - 1 - c : c);
  if (i >= static_cast<long long>(planes) * n) return -1;
  const long long gsz = static_cast<long long>(group_heads) * n;
  const long long grp = i / gsz;
  const long long r = i - grp * gsz;
  const int h0 = static_cast<int>(grp * group_heads);
  const int hg = planes - h0 < group_heads ? planes - h0 : group_heads;
  const int t = static_cast<int>(r / hg);
  *plane = h0 + static_cast<int>(r - static_cast<long long>(t) * hg);
  return n - 1 - t;
}

// Ring of per-item state in the forward kernel (O-staged barriers, the
// producer's record of where each item's O is staged): items whose O waits in
// a V stage for its TMA store number at most VST + 1 <= kItemRing.
constexpr int kItemRing = 8;

struct SimtParams {
  const float *q, *k, *v;
  float *o, *lse;
  unsigned *status;
  int B, H, Nq, Nk, d;
  int n_qtiles;
  float scale;
  int causal;
  int num_sms;  // SMs of the device (chooses the kernel's work split)
};

// Tensor-core forward for one (head dim, input type); causal chosen inside.
// klo: the fp32 path's staged K_lo map (p.kv_staged), else unused (any valid
// map).  Returns the launch's cudaError_t.
cudaError_t launch_tc_bf16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s);
cudaError_t launch_tc_bf16_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                                int B, int causal, cudaStream_t s);
cudaError_t launch_tc_f32_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                              const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                              int B, int causal, cudaStream_t s);
cudaError_t launch_tc_f32_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s);
// fp32 inputs with staged operands: k and klo are the bf16 halves of the
// split K (the scores as three bf16 products).
cudaError_t launch_tc_f32s_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s);
cudaError_t launch_tc_f32s_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                                int B, int causal, cudaStream_t s);

cudaError_t launch_tc_f16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                              const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                              int B, int causal, cudaStream_t s);
cudaError_t launch_tc_f16_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s);
cudaError_t launch_tc_bf16_d256(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                                int B, int causal, cudaStream_t s);
cudaError_t launch_tc_f16_d256(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s);

// Merge of the split-mode chunks into o (dtype: bf16, f16 or f32) and lse.
cudaError_t launch_splitkv_combine(const float *ws_o, const float *ws_lse, void *o, float *lse,
                                   int BH, int Nq, int d, int n_ktiles, int nsp, int causal,
                                   int dtype, unsigned *status, cudaStream_t s);

cudaError_t launch_simt(const SimtParams &p, int B, cudaStream_t s);

// fp32 staging pre-pass: kr = bf16(k) and kl = bf16(k - kr) (bf16 arrays in
// k's layout), vt[bh][x][n] = tf32(v[bh][n][x]) for n < Nk and 0 for
// Nk <= n < nk_pad.
cudaError_t launch_stage_f32(const float *k, const float *v, __nv_bfloat16 *kr,
                             __nv_bfloat16 *kl, float *vt, int BH, int Nk, int nk_pad, int d,
                             cudaStream_t s);

// ------------------------------------------------------------------ backward
// Tensor-core backward: one CTA per (key tile, head, batch).  The TMA maps
// view q/dO as [B*H, Nq, d] and k/v as [B*H, Nk, d] (16-bit).
struct BwdParams {
  float *dq_acc;                  // [B*H][Nq][d] fp32, zeroed by the prep kernel
  const float *lse2;              // [B*H][Nq_pad]: LSE * log2(e); +inf on padded rows
  const float *dd;                // [B*H][Nq_pad]: D = rowsum(dO * O); 0 on padded rows
  void *dk, *dv;                  // [B*H][Nk][d], input type
  unsigned *status;
  int H, Nq, Nk, Nq_pad;          // Nq_pad = 128 * n_qtiles
  int n_qtiles, n_ktiles;
  float scale;                    // signed softmax scale
  float scale_log2;               // scale * log2(e), signed
  unsigned long long wait_limit_ns;
  int d_io = 0;                   // head dim in memory when below the kernel's D (0 = D)
  // Variable-length batches (token-major [total, H, d]; LSE/D rows laid out
  // [H][B][Nq_pad]): device offsets of B+1 entries each, or null.
  const int *cu_q = nullptr;
  const int *cu_k = nullptr;
  int total_q = 0, total_k = 0;
  // Elements of dq_acc, of lse2 (= of dd) and of dK (= of dV), for the debug
  // build's index checks.
  long long dq_elems = 0, row_elems = 0, kv_elems = 0;
};

cudaError_t launch_bwd_bf16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                                cudaStream_t s);
cudaError_t launch_bwd_bf16_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                 const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                                 cudaStream_t s);
cudaError_t launch_bwd_f16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                               cudaStream_t s);
cudaError_t launch_bwd_f16_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                                cudaStream_t s);

// fp32 backward on the CUDA cores (FA_DTYPE_F32 and FA_DTYPE_F32_SIMT, head
// dim 1..128): dd receives D = rowsum(dO * O) per query row (B*H*Nq floats),
// dq is zeroed and then accumulated with atomics, dk and dv are written.
cudaError_t launch_bwd_simt(const float *q, const float *k, const float *v, const float *o,
                            const float *lse, const float *dout, float *dq, float *dk, float *dv,
                            float *dd, int B, int H, int Nq, int Nk, int d, float scale,
                            int causal, unsigned *status, cudaStream_t s);

// D = rowsum(dO * O) and LSE * log2(e) per padded row, and dq_acc zeroed.
cudaError_t launch_bwd_prep(const void *o, const void *dout, const float *lse, float *lse2,
                            float *dd, float *dq_acc, int BH, int Nq, int Nq_pad, int d, int half,
                            cudaStream_t s);
// The same for variable-length batches: rows [H][B][Nq_pad] of lse2 and dd,
// dq_acc token-major [total_q, H, d].
cudaError_t launch_bwd_prep_varlen(const void *o, const void *dout, const float *lse, float *lse2,
                                   float *dd, float *dq_acc, const int *cu_q, int B, int H,
                                   int total_q, int Nq_pad, int d, int half, cudaStream_t s);
// dq (rows of d elements) = dq_acc rounded to the input type; total_q > 0
// selects the variable-length layouts (token-major dq, [H][total_q] rows).
cudaError_t launch_bwd_convert(const float *dq_acc, void *dq, long long rows, int d, int H,
                               int total_q, int half, cudaStream_t s);

}  // namespace fa
