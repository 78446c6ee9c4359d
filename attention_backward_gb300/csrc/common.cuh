// Workspace layout, device error codes and the tile schedule, shared by the
// host entry points and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>

namespace ab {

constexpr int64_t kHeaderBytes = 256;

// Default limit of one bounded wait inside a kernel.
constexpr uint64_t kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Header at the start of every workspace.
struct WsHeader {
  int err;           // first device error code (0: none)
  int tile_counter;  // scratch for persistent schedulers
  int pad[62];
};

struct WsLayout {
  int64_t lse2_off, delta_off, dq_off, dkv_off, total;
};

__host__ __device__ inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int64_t B, int64_t S, int64_t H, int64_t Dq, int64_t dkv_elems) {
  WsLayout L;
  const int64_t rows = B * H * S;
  L.lse2_off = kHeaderBytes;
  L.delta_off = L.lse2_off + round_up(rows * 4, 256);
  L.dq_off = L.delta_off + round_up(rows * 4, 256);
  L.dkv_off = L.dq_off + round_up(B * S * H * Dq * 4, 256);
  L.total = L.dkv_off + round_up(dkv_elems * 4, 256);
  return L;
}

// Device error codes: which bounded wait ran out.
enum DeviceError : int {
  kErrNone = 0,
  kErrWaitKV = 0x101,
  kErrWaitStageEmpty = 0x102,
  kErrWaitStageFull = 0x103,
  kErrWaitS = 0x104,
  kErrWaitP = 0x105,
  kErrWaitDP = 0x107,
  kErrWaitDS = 0x108,
  kErrWaitDSFree = 0x109,
  kErrWaitSFree = 0x10A,
  kErrWaitDQFull = 0x10B,
  kErrWaitDQEmpty = 0x10C,
  kErrWaitDKV = 0x10D,
  kErrWaitTile = 0x10E,
  kErrWaitKVFree = 0x10F,
  kErrWaitStage = 0x110,
  kErrWaitDKVFree = 0x111,
  kErrWaitTail = 0x112,
  kErrAlign = 0x1FE,
  kErrSelftest = 0x1FF,
  kErrSparseBase = 0x200,
};

__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

// Query blocks [lo, hi) (blocks of ``bq`` query positions) that the key tile
// [k0, min(k0 + bk, klen)) of a row of ``klen`` keys and ``qlen`` queries must
// visit, query i standing at key position i + off (off = klen - qlen for a
// dense row whose lengths differ, else 0).  Key j is visible to query i iff
// j <= i + off (causal or window) and i + off < j + W (window W > 0).
__host__ __device__ inline void query_block_range_qk(int k0, int bk, int klen, int qlen, int off, int causal,
                                                     int window, int bq, int* lo, int* hi) {
  const int k1 = imin(k0 + bk, klen);
  int64_t q_start = 0, q_end = qlen;
  if (causal || window > 0) q_start = static_cast<int64_t>(k0) - off;
  if (q_start < 0) q_start = 0;
  if (window > 0) {
    const int64_t e = static_cast<int64_t>(k1) - 1 - off + window;
    q_end = e < qlen ? e : qlen;
  }
  if (k0 >= klen || q_start >= q_end) {
    *lo = *hi = 0;
    return;
  }
  *lo = static_cast<int>(q_start / bq);
  *hi = static_cast<int>((q_end + bq - 1) / bq);
}

// The same for equal query and key lengths (the sequence-local positions of a
// packed sequence or of a dense row with Sk == Sq).
__host__ __device__ inline void query_block_range(int k0, int bk, int len, int causal, int window, int bq, int* lo,
                                                  int* hi) {
  query_block_range_qk(k0, bk, len, len, 0, causal, window, bq, lo, hi);
}

// Sequence bounds of batch row b / packed sequence n, clamped to [0, S].
__host__ __device__ inline int clamp_pos(int x, int S) { return x < 0 ? 0 : (x > S ? S : x); }

// Rows [r0, r1) of a block of ``rows`` positions starting at position ``base``
// of a packed batch that lie in [tail0, S): past the last sequence but inside
// the tensor, so a TMA load reads whatever the caller left there (rows past S
// read zeros).  Empty (r0 >= r1) when the block does not reach the tail.
__host__ __device__ inline void tail_rows(int base, int rows, int tail0, int S, int* r0, int* r1) {
  const int a = tail0 - base, e = S - base;
  *r0 = a < 0 ? 0 : a;
  *r1 = e < rows ? e : rows;
}

}  // namespace ab
