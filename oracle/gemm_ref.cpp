// CPU oracle for the dense GEMM D[l] = alpha * A[l] * B[l] + beta * C[l].
//
// TEST INFRASTRUCTURE. Only the test suite, the package's smoke entry and the
// benchmark's CPU-baseline leg may load this library. The product path never
// calls it; it shares no source, header or helper with the CUDA library.
//
// What it computes is the plain definition of the GEMM that the cited
// CUTLASS kernels implement: the epilogue of "sm90_gemm_tma_warpspecialized_cooperative.hpp"
// (the C-load collective and `collective_epilogue.store`) forms
// alpha * accumulator + beta * C per output element, where the accumulator is
// the sum over k of A(m,k) * B(k,n) for one (m, n, l) of the MNKL problem
// shape. Written out element by element, in fp64, k summed in increasing order:
//
//   ref[l,i,j] = double(alpha) * sum_k double(A[l,i,k]) * double(B[l,k,j])
//              + double(beta) * double(C[l,i,j])          (only when beta != 0)
//
// Layouts (packed batches): A is L x M x K row-major; B is column-major K x N
// per batch, stored as L x N x K with K contiguous; C is L x M x N row-major.
// Inputs are raw bf16 bit patterns; the result is left in fp64 (not rounded).
//
// Readings where those sources are silent: with beta == 0 the C term is skipped,
// not multiplied by zero (so C may be absent); alpha and beta are fp32 values
// widened to fp64.
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// bf16 is the upper half of an IEEE binary32; widening to fp64 is exact.
double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

struct Problem {
  const uint16_t* A;
  const uint16_t* B;
  const uint16_t* C;
  double* out;
  int64_t M, N, K, L;
  double alpha, beta;
  const int64_t* rows;
};

// One output row: r indexes `rows`, which holds global row ids l*M + i.
void one_row(const Problem& p, int64_t r) {
  const int64_t g = p.rows[r];
  const int64_t l = g / p.M;
  const int64_t i = g % p.M;
  for (int64_t j = 0; j < p.N; ++j) {
    double s = 0.0;
    for (int64_t k = 0; k < p.K; ++k) {
      const double a = bf16_to_double(p.A[(l * p.M + i) * p.K + k]);
      const double b = bf16_to_double(p.B[(l * p.N + j) * p.K + k]);
      s += a * b;
    }
    double v = p.alpha * s;
    if (p.beta != 0.0) v += p.beta * bf16_to_double(p.C[(l * p.M + i) * p.N + j]);
    p.out[r * p.N + j] = v;
  }
}

}  // namespace

extern "C" {

// Computes the requested output rows in fp64.
//   rows[0..nrows)  global row ids l*M + i, each in [0, L*M)
//   out             nrows x N doubles, row r holds output row rows[r]
//   threads         worker threads (<= 0 means 1); rows are dealt round-robin
// Returns 0, or -1 on a bad argument (null pointer, C absent with beta != 0,
// negative size, row id out of range).
int oracle_gemm_rows(const uint16_t* A, const uint16_t* B, const uint16_t* C,
                     double* out, int64_t M, int64_t N, int64_t K, int64_t L,
                     float alpha, float beta, const int64_t* rows,
                     int64_t nrows, int threads) {
  if (M < 0 || N < 0 || K < 0 || L < 0 || nrows < 0) return -1;
  if (nrows == 0 || N == 0) return 0;
  if (!out || !rows) return -1;
  if (K > 0 && (!A || !B)) return -1;
  if (beta != 0.0f && !C) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= L * M) return -1;

  Problem p{A, B, C, out, M, N, K, L, static_cast<double>(alpha),
            static_cast<double>(beta), rows};
  if (threads < 1) threads = 1;
  if (threads > nrows) threads = static_cast<int>(nrows);
  if (threads == 1) {
    for (int64_t r = 0; r < nrows; ++r) one_row(p, r);
    return 0;
  }
  std::vector<std::thread> pool;
  pool.reserve(threads);
  for (int t = 0; t < threads; ++t) {
    pool.emplace_back([&p, t, threads, nrows]() {
      for (int64_t r = t; r < nrows; r += threads) one_row(p, r);
    });
  }
  for (auto& th : pool) th.join();
  return 0;
}

}  // extern "C"
