// Ring all-reduce ORACLE — test infrastructure only.
//
// A plain, deliberately slow CPU simulation of the ring schedule: one
// std::thread per rank, one unbounded FIFO channel from each rank to its right
// neighbour, and the reduce-scatter / all-gather index arithmetic exactly as
// the tirogla.com page "Ring all-reduce" (section "How it works") states it:
//
//   reduce-scatter, step s = 0..N-2: rank r sends chunk (r - s) mod N to r+1,
//     receives chunk (r - s - 1) mod N from r-1 and combines it into its copy;
//     afterwards rank r holds the complete reduction of chunk (r + 1) mod N.
//   all-gather, step s = 0..N-2: rank r sends chunk (r + 1 - s) mod N,
//     receives chunk (r - s) mod N and overwrites its copy.
//
// Chunk c covers elements [c*len/N, (c+1)*len/N) with floor division, so
// chunks may differ in length by one element and may be empty (same page,
// section "Code": the self-test uses len = 1003 over 5 ranks on purpose).
//
// Only tests/, the package's smoke check and the bench's CPU-baseline leg use
// this file. It shares no code with the CUDA library: its own chunk bounds,
// its own IEEE round-to-nearest-even conversions, its own reduction ops.
//
// Precision (the pages fix it): every hop is rounded to the buffer dtype.
// fp32 hops are plain fp32 arithmetic; fp16/bf16 hops widen both operands to
// fp32 (exact), apply the op in fp32 and round once to the dtype (RNE);
// int32 hops use two's-complement wrap. avg = the ring sum, then one multiply
// by inv_n = 1.0f/N (fp32) rounded to the dtype; int32 avg = wrapped sum
// divided by N with C truncation.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared -pthread
// (no -ffast-math: subnormals, NaN and signed zero must follow IEEE 754).

#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <deque>
#include <mutex>
#include <thread>
#include <vector>

namespace {

enum Dtype { F32 = 0, F16 = 1, BF16 = 2, I32 = 3 };
enum Op { SUM = 0, AVG = 1, MIN = 2, MAX = 3, PROD = 4 };
enum Status {
  ORACLE_OK = 0,
  ORACLE_INVALID = 1,
  ORACLE_UNSUPPORTED = 2,
  ORACLE_TIMEOUT = 3,   // a recv saw no message within the time limit
  ORACLE_PROTOCOL = 4,  // a message of the wrong length arrived
  ORACLE_FAULTED = 5,   // this rank was told to stop (host fault injection)
};

constexpr int kMaxRanks = 64;

size_t elem_size(int dt) {
  switch (dt) {
    case F32: return 4;
    case F16: return 2;
    case BF16: return 2;
    case I32: return 4;
    default: return 0;
  }
}

// ---- chunk bounds (tirogla "Ring all-reduce", section "Code") -------------
// c*len/n with floor division, computed in 128 bits so no product overflows.
uint64_t chunk_begin(uint64_t c, uint64_t n, uint64_t len) {
  return (uint64_t)(((unsigned __int128)c * len) / n);
}
uint64_t chunk_end(uint64_t c, uint64_t n, uint64_t len) { return chunk_begin(c + 1, n, len); }
int mod(long a, long n) { return (int)(((a % n) + n) % n); }

// ---- IEEE 754 narrow formats, written from the standard's definition -------
// A binary format with p significand bits (hidden bit included) and exponent
// bias `bias`. Narrow values are decoded exactly into fp32 (every fp16 and
// bf16 value is an fp32 value).
struct Narrow {
  int p;     // significand bits incl. hidden: fp16 11, bf16 8
  int ebits; // exponent field width: fp16 5, bf16 8
  int bias;  // fp16 15, bf16 127
};
constexpr Narrow kF16{11, 5, 15};
constexpr Narrow kBF16{8, 8, 127};

float narrow_to_f32(uint16_t h, const Narrow& f) {
  const int fbits = f.p - 1;
  const uint32_t sign = (h >> (fbits + f.ebits)) & 1u;
  const uint32_t e = (h >> fbits) & ((1u << f.ebits) - 1u);
  const uint32_t frac = h & ((1u << fbits) - 1u);
  float v;
  if (e == (1u << f.ebits) - 1u) {
    v = frac ? NAN : INFINITY;
  } else if (e == 0) {
    // subnormal: frac * 2^(1 - bias - fbits)
    v = std::ldexp((float)frac, 1 - f.bias - fbits);
  } else {
    v = std::ldexp((float)(frac | (1u << fbits)), (int)e - f.bias - fbits);
  }
  return sign ? -v : v;
}

// Round an fp32 value to the narrow format, round-to-nearest, ties to even.
// The value is taken apart as an integer significand m times 2^q, the quantum
// of the target binade is found, and the integer is rounded at that quantum.
uint16_t f32_to_narrow(float x, const Narrow& f) {
  uint32_t bits;
  std::memcpy(&bits, &x, 4);
  const int fbits = f.p - 1;
  const uint16_t sign = (uint16_t)((bits >> 31) << (fbits + f.ebits));
  const uint32_t e32 = (bits >> 23) & 0xffu;
  const uint32_t m32 = bits & 0x7fffffu;
  const uint16_t exp_all_ones = (uint16_t)(((1u << f.ebits) - 1u) << fbits);
  if (e32 == 0xffu) {
    if (m32 == 0) return sign | exp_all_ones;               // infinity
    return sign | exp_all_ones | (uint16_t)(1u << (fbits - 1));  // quiet NaN
  }
  if (e32 == 0 && m32 == 0) return sign;                    // signed zero
  uint64_t m = e32 ? (m32 | 0x800000u) : m32;               // value = m * 2^q
  int q = e32 ? (int)e32 - 150 : -149;
  int msb = 63 - __builtin_clzll(m);                        // binade exponent = q + msb
  const int min_quantum = 1 - f.bias - fbits;               // subnormal spacing
  int tq = q + msb - fbits;                                 // quantum of the binade
  if (tq < min_quantum) tq = min_quantum;
  int shift = tq - q;
  uint64_t r;
  if (shift <= 0) {
    r = m << (-shift);
  } else if (shift > 40) {
    r = 0;  // far below half a quantum
  } else {
    r = m >> shift;
    const uint64_t rem = m & ((1ull << shift) - 1ull);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (r & 1ull))) r += 1;
  }
  if (r == 0) return sign;
  // value = r * 2^tq, r < 2^p (or == 2^p after a carry)
  if (r >= (1ull << f.p)) {  // carry out of the significand
    r >>= 1;
    tq += 1;
  }
  if (r < (1ull << fbits)) {
    // only possible at the minimum quantum: a subnormal
    return sign | (uint16_t)r;
  }
  const int efield = tq + fbits + f.bias;
  if (efield >= (1 << f.ebits) - 1) return sign | exp_all_ones;  // overflow to inf
  return sign | (uint16_t)((uint32_t)efield << fbits) | (uint16_t)(r - (1ull << fbits));
}

// ---- IEEE 754-2019 minimum / maximum: NaN propagates, -0 < +0 -------------
float ieee_minimum(float a, float b) {
  if (std::isnan(a)) return a;
  if (std::isnan(b)) return b;
  if (a < b) return a;
  if (b < a) return b;
  return std::signbit(a) ? a : b;  // equal: only the sign of zero can differ
}
float ieee_maximum(float a, float b) {
  if (std::isnan(a)) return a;
  if (std::isnan(b)) return b;
  if (a > b) return a;
  if (b > a) return b;
  return std::signbit(a) ? b : a;
}

float f32_op(int op, float a, float b) {
  switch (op) {
    case SUM:
    case AVG: return a + b;
    case PROD: return a * b;
    case MIN: return ieee_minimum(a, b);
    case MAX: return ieee_maximum(a, b);
  }
  return NAN;
}

// One ring hop on one element: `partial` is the incoming message value (the
// left operand), `local` is this rank's own value. Storage-typed in and out.
void hop(int dt, int op, const uint8_t* partial, const uint8_t* local, uint8_t* out) {
  switch (dt) {
    case F32: {
      float a, b;
      std::memcpy(&a, partial, 4);
      std::memcpy(&b, local, 4);
      float r = f32_op(op, a, b);
      std::memcpy(out, &r, 4);
      return;
    }
    case F16:
    case BF16: {
      const Narrow& f = (dt == F16) ? kF16 : kBF16;
      uint16_t ha, hb;
      std::memcpy(&ha, partial, 2);
      std::memcpy(&hb, local, 2);
      const float a = narrow_to_f32(ha, f), b = narrow_to_f32(hb, f);
      uint16_t r;
      if (op == MIN || op == MAX) {
        // the result is one of the operands: keep its bits (no rounding)
        const float m = f32_op(op, a, b);
        if (std::isnan(m)) r = std::isnan(a) ? ha : hb;
        else if (std::memcmp(&m, &a, 4) == 0) r = ha;
        else r = hb;
      } else {
        r = f32_to_narrow(f32_op(op, a, b), f);
      }
      std::memcpy(out, &r, 2);
      return;
    }
    case I32: {
      uint32_t a, b, r = 0;
      std::memcpy(&a, partial, 4);
      std::memcpy(&b, local, 4);
      int32_t sa, sb;
      std::memcpy(&sa, &a, 4);
      std::memcpy(&sb, &b, 4);
      switch (op) {
        case SUM:
        case AVG: r = a + b; break;   // wraps mod 2^32
        case PROD: r = a * b; break;  // wraps mod 2^32
        case MIN: r = (uint32_t)(sa < sb ? sa : sb); break;
        case MAX: r = (uint32_t)(sa > sb ? sa : sb); break;
      }
      std::memcpy(out, &r, 4);
      return;
    }
  }
}

// The avg epilogue, applied once by the rank that finished the chunk
// (bitfern.com "AllReduce Explained", section on data-parallel training:
// gradients summed, then divided by the number of workers).
void avg_epilogue(int dt, int n, uint8_t* v) {
  const float inv_n = 1.0f / (float)n;
  switch (dt) {
    case F32: {
      float a;
      std::memcpy(&a, v, 4);
      a = a * inv_n;
      std::memcpy(v, &a, 4);
      return;
    }
    case F16:
    case BF16: {
      const Narrow& f = (dt == F16) ? kF16 : kBF16;
      uint16_t h;
      std::memcpy(&h, v, 2);
      h = f32_to_narrow(narrow_to_f32(h, f) * inv_n, f);
      std::memcpy(v, &h, 2);
      return;
    }
    case I32: {
      int32_t a;
      std::memcpy(&a, v, 4);
      a = a / n;  // C division: truncates toward zero
      std::memcpy(v, &a, 4);
      return;
    }
  }
}

// ---- channels --------------------------------------------------------------
// An unbounded FIFO: send never blocks (a blocking send before recv can
// deadlock; infra-guide "Collective communication primitives", section 2),
// recv waits at most `timeout_ms` and reports failure instead of hanging.
class Channel {
 public:
  void send(std::vector<uint8_t> msg) {
    {
      std::lock_guard<std::mutex> lk(m_);
      q_.push_back(std::move(msg));
    }
    cv_.notify_one();
  }
  bool recv(std::vector<uint8_t>& out, int timeout_ms) {
    std::unique_lock<std::mutex> lk(m_);
    if (!cv_.wait_for(lk, std::chrono::milliseconds(timeout_ms), [&] { return !q_.empty(); }))
      return false;
    out = std::move(q_.front());
    q_.pop_front();
    return true;
  }

 private:
  std::mutex m_;
  std::condition_variable cv_;
  std::deque<std::vector<uint8_t>> q_;
};

struct Ring {
  int n = 0;
  uint64_t len = 0;
  int dt = 0, op = 0;
  size_t es = 0;
  int timeout_ms = 0;
  std::vector<Channel> into;        // into[r]: the channel from rank r-1 to rank r
  uint64_t* bytes_sent = nullptr;   // [n] or null
  uint8_t* snapshots = nullptr;     // [2(n-1)][n][len] elements or null
  int fault_rank = -1, fault_step = -1;
  std::vector<int> status;

  explicit Ring(int n_) : n(n_), into(n_), status(n_, ORACLE_OK) {}

  uint8_t* chunk_ptr(uint8_t* d, int c) const { return d + chunk_begin(c, n, len) * es; }
  size_t chunk_bytes(int c) const { return (chunk_end(c, n, len) - chunk_begin(c, n, len)) * es; }

  void send_chunk(int r, const uint8_t* d, int c) {
    const size_t nb = chunk_bytes(c);
    const uint8_t* p = d + chunk_begin(c, n, len) * es;
    into[(r + 1) % n].send(std::vector<uint8_t>(p, p + nb));
    if (bytes_sent) bytes_sent[r] += nb;
  }
  // returns false (and records why) if the message does not arrive or is malformed
  bool recv_chunk(int r, int c, std::vector<uint8_t>& in) {
    if (!into[r].recv(in, timeout_ms)) {
      status[r] = ORACLE_TIMEOUT;
      return false;
    }
    if (in.size() != chunk_bytes(c)) {
      status[r] = ORACLE_PROTOCOL;
      return false;
    }
    return true;
  }
  void snapshot(int step, int r, const uint8_t* d) {
    if (!snapshots) return;
    std::memcpy(snapshots + ((size_t)step * n + r) * len * es, d, len * es);
  }
  bool faulted(int r, int step) {
    if (r == fault_rank && step == fault_step) {
      status[r] = ORACLE_FAULTED;
      return true;
    }
    return false;
  }

  // Reduce-scatter phase on rank r's working copy d. Returns false on failure.
  bool reduce_scatter_phase(int r, uint8_t* d) {
    std::vector<uint8_t> in;
    for (int s = 0; s + 1 < n; ++s) {
      if (faulted(r, s)) return false;
      const int send_c = mod((long)r - s, n);
      const int recv_c = mod((long)r - s - 1, n);
      send_chunk(r, d, send_c);
      if (!recv_chunk(r, recv_c, in)) return false;
      uint8_t* dst = chunk_ptr(d, recv_c);
      const size_t cnt = in.size() / es;
      for (size_t k = 0; k < cnt; ++k) hop(dt, op, &in[k * es], dst + k * es, dst + k * es);
      snapshot(s, r, d);
    }
    // rank r now owns the complete chunk (r + 1) mod N; avg finishes it here
    if (op == AVG) {
      const int own = (r + 1) % n;
      uint8_t* p = chunk_ptr(d, own);
      const size_t cnt = chunk_bytes(own) / es;
      for (size_t k = 0; k < cnt; ++k) avg_epilogue(dt, n, p + k * es);
    }
    return true;
  }

  // All-gather phase: first_send is the chunk a rank sends at step 0
  // ((r+1) after a reduce-scatter, r for a standalone all-gather).
  bool all_gather_phase(int r, uint8_t* d, int shift, int step_base) {
    std::vector<uint8_t> in;
    for (int s = 0; s + 1 < n; ++s) {
      if (faulted(r, step_base + s)) return false;
      const int send_c = mod((long)r + shift - s, n);
      const int recv_c = mod((long)r + shift - s - 1, n);
      send_chunk(r, d, send_c);
      if (!recv_chunk(r, recv_c, in)) return false;
      if (!in.empty()) std::memcpy(chunk_ptr(d, recv_c), in.data(), in.size());
      snapshot(step_base + s, r, d);
    }
    return true;
  }

  int result() const {
    int worst = ORACLE_OK;
    for (int s : status)
      if (s != ORACLE_OK && (worst == ORACLE_OK || s == ORACLE_TIMEOUT)) worst = s;
    return worst;
  }
};

// ---- a full mesh of channels, for the algorithms that talk to partners ----
struct Mesh {
  int n;
  std::vector<Channel> chan;  // chan[src * n + dst]
  int timeout_ms;
  uint64_t* bytes_sent;
  std::vector<int> status;
  Mesh(int n_, int timeout, uint64_t* bytes)
      : n(n_), chan((size_t)n_ * n_), timeout_ms(timeout), bytes_sent(bytes), status(n_, ORACLE_OK) {}
  void send(int src, int dst, const uint8_t* p, size_t nb) {
    chan[(size_t)src * n + dst].send(std::vector<uint8_t>(p, p + nb));
    if (bytes_sent) bytes_sent[src] += nb;
  }
  bool recv(int src, int dst, std::vector<uint8_t>& in, size_t want) {
    if (!chan[(size_t)src * n + dst].recv(in, timeout_ms)) {
      status[dst] = ORACLE_TIMEOUT;
      return false;
    }
    if (in.size() != want) {
      status[dst] = ORACLE_PROTOCOL;
      return false;
    }
    return true;
  }
  int result() const {
    for (int s : status)
      if (s != ORACLE_OK) return s;
    return ORACLE_OK;
  }
};

// Rabenseifner's all-reduce for a power-of-two number of ranks (tirogla.com
// "Ring all-reduce", "How it works", cost model: recursive-halving
// reduce-scatter followed by recursive-doubling all-gather). Halving step with
// distance d = N/2, N/4, ..., 1: rank r and its partner r XOR d split their
// current range in two; the rank whose d bit is clear keeps the lower half.
// Each sends the half it gives up and combines the half it keeps with the
// partner's copy, the lower rank's value on the left. The owner of a range
// finishes avg on it; doubling then returns the halves in reverse order.
void rabenseifner_rank(Mesh& M, int r, uint8_t* d, uint64_t len, int dt, int op, size_t es) {
  const int n = M.n;
  uint64_t lo = 0, hi = len;
  std::vector<uint64_t> los, his;
  std::vector<uint8_t> in;
  for (int dist = n / 2; dist >= 1; dist /= 2) {
    const int p = r ^ dist;
    const uint64_t mid = lo + (hi - lo) / 2;
    const bool lower = (r & dist) == 0;
    const uint64_t keep_lo = lower ? lo : mid, keep_hi = lower ? mid : hi;
    const uint64_t give_lo = lower ? mid : lo, give_hi = lower ? hi : mid;
    los.push_back(lo);
    his.push_back(hi);
    M.send(r, p, d + give_lo * es, (give_hi - give_lo) * es);
    if (!M.recv(p, r, in, (keep_hi - keep_lo) * es)) return;
    for (uint64_t k = 0; k < keep_hi - keep_lo; ++k) {
      uint8_t* mine = d + (keep_lo + k) * es;
      const uint8_t* theirs = &in[k * es];
      if (lower) hop(dt, op, mine, theirs, mine);
      else hop(dt, op, theirs, mine, mine);
    }
    lo = keep_lo;
    hi = keep_hi;
  }
  if (op == AVG)
    for (uint64_t k = lo; k < hi; ++k) avg_epilogue(dt, n, d + k * es);
  for (int dist = 1, step = (int)los.size() - 1; dist < n; dist *= 2, --step) {
    const int p = r ^ dist;
    const uint64_t plo = los[step], phi = his[step];
    const uint64_t mid = plo + (phi - plo) / 2;
    const bool lower = (r & dist) == 0;
    const uint64_t other_lo = lower ? mid : plo, other_hi = lower ? phi : mid;
    M.send(r, p, d + lo * es, (hi - lo) * es);
    if (!M.recv(p, r, in, (other_hi - other_lo) * es)) return;
    if (!in.empty()) std::memcpy(d + other_lo * es, in.data(), in.size());
    lo = plo;
    hi = phi;
  }
}

// A binary tree laid over a sequence of ranks in order: the middle position
// is the root, the two halves its subtrees. parent[] / left[] / right[] by rank.
struct InorderTree {
  std::vector<int> parent, left, right;
  int root = -1;
  InorderTree(const std::vector<int>& seq) : parent(seq.size(), -1), left(seq.size(), -1), right(seq.size(), -1) {
    root = build(seq, 0, (int)seq.size() - 1, -1);
  }
  int build(const std::vector<int>& seq, int lo, int hi, int par) {
    if (lo > hi) return -1;
    const int m = (lo + hi) / 2, v = seq[m];
    parent[v] = par;
    left[v] = build(seq, lo, m - 1, v);
    right[v] = build(seq, m + 1, hi, v);
    return v;
  }
};

// Double binary tree (tirogla.com "Ring all-reduce", cost model; NCCL's tree
// since 2.4): two binary trees, each reducing half of the buffer up to its
// root and broadcasting the result back down. Tree A is the in-order tree over
// ranks 0..N-1 and reduces chunks [0, N/2); tree B is the in-order tree over
// ranks N-1..0 and reduces chunks [N/2, N). A node folds in order: its left
// subtree's partial, its own value, its right subtree's partial.
void tree_rank(Mesh& M, int r, uint8_t* d, uint64_t len, int dt, int op, size_t es) {
  const int n = M.n;
  std::vector<int> fwd(n), bwd(n);
  for (int i = 0; i < n; ++i) fwd[i] = i, bwd[i] = n - 1 - i;
  const uint64_t split = chunk_begin(n / 2, n, len);
  std::vector<uint8_t> in;
  for (int t = 0; t < 2; ++t) {
    const InorderTree T(t == 0 ? fwd : bwd);
    const uint64_t lo = t == 0 ? 0 : split, hi = t == 0 ? split : len;
    const size_t nb = (hi - lo) * es;
    uint8_t* mine = d + lo * es;
    if (T.left[r] >= 0) {  // partial of the left subtree, then own value on the right
      if (!M.recv(T.left[r], r, in, nb)) return;
      for (uint64_t k = 0; k < hi - lo; ++k) hop(dt, op, &in[k * es], mine + k * es, mine + k * es);
    }
    if (T.right[r] >= 0) {  // then the right subtree's partial on the right
      if (!M.recv(T.right[r], r, in, nb)) return;
      for (uint64_t k = 0; k < hi - lo; ++k) hop(dt, op, mine + k * es, &in[k * es], mine + k * es);
    }
    if (T.parent[r] >= 0) {
      M.send(r, T.parent[r], mine, nb);
      if (!M.recv(T.parent[r], r, in, nb)) return;  // the result, broadcast down
      if (nb) std::memcpy(mine, in.data(), nb);
    } else if (op == AVG) {
      for (uint64_t k = 0; k < hi - lo; ++k) avg_epilogue(dt, n, mine + k * es);
    }
    if (T.left[r] >= 0) M.send(r, T.left[r], mine, nb);
    if (T.right[r] >= 0) M.send(r, T.right[r], mine, nb);
  }
}

int check_args(uint64_t len, int dt, int op, int n) {
  if (n < 1 || n > kMaxRanks) return ORACLE_INVALID;
  if (elem_size(dt) == 0) return ORACLE_INVALID;
  if (op < SUM || op > PROD) return ORACLE_INVALID;
  if (len > (1ull << 40)) return ORACLE_INVALID;
  return ORACLE_OK;
}

}  // namespace

extern "C" {

int ra_oracle_chunk_range(uint64_t len, int n, int c, uint64_t* begin, uint64_t* end) {
  if (n < 1 || n > kMaxRanks || c < 0 || c >= n || !begin || !end) return ORACLE_INVALID;
  *begin = chunk_begin(c, n, len);
  *end = chunk_end(c, n, len);
  return ORACLE_OK;
}

// All-reduce: send[r] (len elements, host) -> recv[r] (len elements, host),
// which serve as each rank's working copy. recv[r] == send[r] is allowed.
// bytes_sent[n] (optional) counts every message's payload per sending rank.
// snapshots (optional): [2(n-1)][n][len] elements, the state of every rank
// after every step (reduce-scatter steps first, then all-gather steps).
int ra_oracle_allreduce(const void* const* send, void* const* recv, uint64_t len, int dtype,
                        int op, int n, int timeout_ms, uint64_t* bytes_sent, void* snapshots,
                        int fault_rank, int fault_step) {
  int st = check_args(len, dtype, op, n);
  if (st != ORACLE_OK) return st;
  Ring R(n);
  R.len = len;
  R.dt = dtype;
  R.op = op;
  R.es = elem_size(dtype);
  R.timeout_ms = timeout_ms;
  R.bytes_sent = bytes_sent;
  R.snapshots = (uint8_t*)snapshots;
  R.fault_rank = fault_rank;
  R.fault_step = fault_step;
  if (bytes_sent) std::memset(bytes_sent, 0, sizeof(uint64_t) * n);
  for (int r = 0; r < n; ++r)
    if (recv[r] != send[r]) std::memcpy(recv[r], send[r], len * R.es);
  if (n == 1) {
    if (op == AVG)
      for (uint64_t k = 0; k < len; ++k) avg_epilogue(dtype, 1, (uint8_t*)recv[0] + k * R.es);
    return ORACLE_OK;
  }
  std::vector<std::thread> threads;
  for (int r = 0; r < n; ++r) {
    threads.emplace_back([&R, r, recv, n] {
      uint8_t* d = (uint8_t*)recv[r];
      if (!R.reduce_scatter_phase(r, d)) return;
      R.all_gather_phase(r, d, /*shift=*/1, /*step_base=*/n - 1);
    });
  }
  for (auto& t : threads) t.join();
  return R.result();
}

// Reduce-scatter: send[r] holds len elements; recv[r] receives chunk r
// (chunk_end(r) - chunk_begin(r) elements, compact). The reduction of chunk r
// is the ring fold finished by rank r-1, which hands it to rank r as one more
// message (the same move as the first all-gather step).
int ra_oracle_reduce_scatter(const void* const* send, void* const* recv, uint64_t len, int dtype,
                             int op, int n, int timeout_ms, uint64_t* bytes_sent) {
  int st = check_args(len, dtype, op, n);
  if (st != ORACLE_OK) return st;
  Ring R(n);
  R.len = len;
  R.dt = dtype;
  R.op = op;
  R.es = elem_size(dtype);
  R.timeout_ms = timeout_ms;
  R.bytes_sent = bytes_sent;
  if (bytes_sent) std::memset(bytes_sent, 0, sizeof(uint64_t) * n);
  std::vector<std::vector<uint8_t>> work(n);
  for (int r = 0; r < n; ++r)
    work[r].assign((const uint8_t*)send[r], (const uint8_t*)send[r] + len * R.es);
  if (n == 1) {
    if (op == AVG)
      for (uint64_t k = 0; k < len; ++k) avg_epilogue(dtype, 1, work[0].data() + k * R.es);
    if (len) std::memcpy(recv[0], work[0].data(), len * R.es);
    return ORACLE_OK;
  }
  std::vector<std::thread> threads;
  for (int r = 0; r < n; ++r) {
    threads.emplace_back([&R, &work, r, recv, n] {
      uint8_t* d = work[r].data();
      if (!R.reduce_scatter_phase(r, d)) return;
      R.send_chunk(r, d, (r + 1) % n);  // hand the finished chunk to its owner
      std::vector<uint8_t> in;
      if (!R.recv_chunk(r, r, in)) return;
      if (!in.empty()) std::memcpy(recv[r], in.data(), in.size());
    });
  }
  for (auto& t : threads) t.join();
  return R.result();
}

// All-gather: send[r] holds chunk r (compact); recv[r] (len elements)
// receives every chunk at its place. Standalone ring all-gather
// (ramchalamkr.github.io "NCCL Primitives Deep Dive", section 1, ring
// all-gather): at step s rank r sends chunk (r - s), receives (r - s - 1).
int ra_oracle_allgather(const void* const* send, void* const* recv, uint64_t len, int dtype, int n,
                        int timeout_ms, uint64_t* bytes_sent, void* snapshots) {
  int st = check_args(len, dtype, SUM, n);
  if (st != ORACLE_OK) return st;
  Ring R(n);
  R.len = len;
  R.dt = dtype;
  R.op = SUM;
  R.es = elem_size(dtype);
  R.timeout_ms = timeout_ms;
  R.bytes_sent = bytes_sent;
  R.snapshots = (uint8_t*)snapshots;
  if (bytes_sent) std::memset(bytes_sent, 0, sizeof(uint64_t) * n);
  for (int r = 0; r < n; ++r) {
    uint8_t* d = (uint8_t*)recv[r];
    std::memset(d, 0, len * R.es);
    const size_t nb = R.chunk_bytes(r);
    if (nb) std::memcpy(R.chunk_ptr(d, r), send[r], nb);
  }
  if (n == 1) return ORACLE_OK;
  std::vector<std::thread> threads;
  for (int r = 0; r < n; ++r) {
    threads.emplace_back([&R, r, recv] {
      R.all_gather_phase(r, (uint8_t*)recv[r], /*shift=*/0, /*step_base=*/0);
    });
  }
  for (auto& t : threads) t.join();
  return R.result();
}

// All-reduce with a choice of algorithm (order) and accumulation precision.
// order 0 = ring (as ra_oracle_allreduce), 1 = double binary tree,
// 2 = Rabenseifner (power-of-two n only). accum 0 = every hop rounded to the
// dtype; accum 1 = fp16/bf16 partials travel as fp32 messages and the owner
// rounds once, after the avg multiply (tirogla.com "Ring all-reduce",
// "Implementation notes": bf16 with fp32 accumulation at large N); for fp32 and
// int32 buffers accum 1 is the same as accum 0. accum 1 is defined for the
// ring only.
int ra_oracle_allreduce_ex(const void* const* send, void* const* recv, uint64_t len, int dtype, int op,
                           int n, int order, int accum, int timeout_ms, uint64_t* bytes_sent) {
  int st = check_args(len, dtype, op, n);
  if (st != ORACLE_OK) return st;
  if (order < 0 || order > 2 || accum < 0 || accum > 1) return ORACLE_INVALID;
  if (order == 2 && (n & (n - 1))) return ORACLE_UNSUPPORTED;
  if (accum == 1 && order != 0) return ORACLE_UNSUPPORTED;
  const bool narrow = dtype == F16 || dtype == BF16;
  if (order == 0 && (accum == 0 || !narrow))
    return ra_oracle_allreduce(send, recv, len, dtype, op, n, timeout_ms, bytes_sent, nullptr, -1, -1);
  const size_t es = elem_size(dtype);
  if (bytes_sent) std::memset(bytes_sent, 0, sizeof(uint64_t) * n);
  if (order == 0) {
    // ring with fp32 messages: run the reduce-scatter phase on widened copies,
    // round the owned chunk once, then the all-gather phase in the dtype
    const Narrow& f = dtype == F16 ? kF16 : kBF16;
    std::vector<std::vector<float>> w(n, std::vector<float>(len));
    for (int r = 0; r < n; ++r)
      for (uint64_t k = 0; k < len; ++k) w[r][k] = narrow_to_f32(((const uint16_t*)send[r])[k], f);
    if (n == 1) {
      for (uint64_t k = 0; k < len; ++k) {
        float v = w[0][k];
        if (op == AVG) v = v * (1.0f / (float)n);
        ((uint16_t*)recv[0])[k] = f32_to_narrow(v, f);
      }
      return ORACLE_OK;
    }
    Ring rs(n), ag(n);
    rs.len = ag.len = len;
    rs.dt = F32;
    ag.dt = dtype;
    rs.op = ag.op = op;
    rs.es = 4;
    ag.es = es;
    rs.timeout_ms = ag.timeout_ms = timeout_ms;
    rs.bytes_sent = ag.bytes_sent = bytes_sent;
    std::vector<std::thread> threads;
    for (int r = 0; r < n; ++r) {
      threads.emplace_back([&, r] {
        if (!rs.reduce_scatter_phase(r, (uint8_t*)w[r].data())) return;
        const int own = (r + 1) % n;
        uint16_t* out = (uint16_t*)recv[r];
        for (uint64_t k = chunk_begin(own, n, len); k < chunk_end(own, n, len); ++k)
          out[k] = f32_to_narrow(w[r][k], f);
        ag.all_gather_phase(r, (uint8_t*)recv[r], /*shift=*/1, /*step_base=*/0);
      });
    }
    for (auto& t : threads) t.join();
    const int a = rs.result();
    return a != ORACLE_OK ? a : ag.result();
  }
  for (int r = 0; r < n; ++r)
    if (recv[r] != send[r]) std::memcpy(recv[r], send[r], len * es);
  if (n == 1) {
    if (op == AVG)
      for (uint64_t k = 0; k < len; ++k) avg_epilogue(dtype, 1, (uint8_t*)recv[0] + k * es);
    return ORACLE_OK;
  }
  Mesh M(n, timeout_ms, bytes_sent);
  std::vector<std::thread> threads;
  for (int r = 0; r < n; ++r) {
    threads.emplace_back([&, r] {
      if (order == 1) tree_rank(M, r, (uint8_t*)recv[r], len, dtype, op, es);
      else rabenseifner_rank(M, r, (uint8_t*)recv[r], len, dtype, op, es);
    });
  }
  for (auto& t : threads) t.join();
  return M.result();
}

// The plain definition at selected indices, with no message passing: element
// i belongs to chunk c (found by scanning the chunk bounds); its result is the
// left fold x_c, x_{c+1}, ..., x_{c+N-1} (ranks mod N) with every hop rounded,
// then the avg epilogue. out[k] receives the result for element idx[k].
int ra_oracle_fold_at(const void* const* send, uint64_t len, int dtype, int op, int n,
                      const uint64_t* idx, uint64_t m, void* out) {
  int st = check_args(len, dtype, op, n);
  if (st != ORACLE_OK) return st;
  const size_t es = elem_size(dtype);
  for (uint64_t k = 0; k < m; ++k) {
    const uint64_t i = idx[k];
    if (i >= len) return ORACLE_INVALID;
    int c = 0;
    while (!(i >= chunk_begin(c, n, len) && i < chunk_end(c, n, len))) ++c;
    uint8_t acc[4];
    std::memcpy(acc, (const uint8_t*)send[c] + i * es, es);
    for (int j = 1; j < n; ++j) {
      const int r = (c + j) % n;
      hop(dtype, op, acc, (const uint8_t*)send[r] + i * es, acc);
    }
    if (op == AVG) avg_epilogue(dtype, n, acc);
    std::memcpy((uint8_t*)out + k * es, acc, es);
  }
  return ORACLE_OK;
}

// Element-wise hop, exposed so tests can pin the rounding of one ring step.
int ra_oracle_hop(int dtype, int op, const void* partial, const void* local, void* out, uint64_t m) {
  if (elem_size(dtype) == 0 || op < SUM || op > PROD) return ORACLE_INVALID;
  const size_t es = elem_size(dtype);
  for (uint64_t k = 0; k < m; ++k)
    hop(dtype, op, (const uint8_t*)partial + k * es, (const uint8_t*)local + k * es,
        (uint8_t*)out + k * es);
  return ORACLE_OK;
}

// fp32 -> fp16/bf16 (RNE) and back, exposed for the conversion pins.
int ra_oracle_round(int dtype, const float* in, uint16_t* out, uint64_t m) {
  if (dtype != F16 && dtype != BF16) return ORACLE_INVALID;
  const Narrow& f = dtype == F16 ? kF16 : kBF16;
  for (uint64_t k = 0; k < m; ++k) out[k] = f32_to_narrow(in[k], f);
  return ORACLE_OK;
}
int ra_oracle_widen(int dtype, const uint16_t* in, float* out, uint64_t m) {
  if (dtype != F16 && dtype != BF16) return ORACLE_INVALID;
  const Narrow& f = dtype == F16 ? kF16 : kBF16;
  for (uint64_t k = 0; k < m; ++k) out[k] = narrow_to_f32(in[k], f);
  return ORACLE_OK;
}

}  // extern "C"
