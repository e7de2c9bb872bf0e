// CPU oracle for submanifold sparse 3D convolution (kernel 3, stride 1, no padding),
// plain C++ for the workloads that are too large for the Python loops.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg. The CUDA library never calls it and shares no code,
// header or table with it.
//
// It computes the same plain definition as ref.py in this directory:
//   S = { (b, z, y, x) -> input row }                      (std::unordered_map)
//   nbr[i, k] = S[(b, z+dz, y+dy, x+dx)] or -1, k = 9(dz+1) + 3(dy+1) + (dx+1),
//               a neighbour outside [0, res)^3 being absent
//   out[i, o] = bias[o] + sum_{k: nbr>=0} sum_c W[o, dz+1, dy+1, dx+1, c] * f[nbr, c]
// accumulated in double from the stored (fp32, or bf16-exact fp32) values.
// Sources: "pixal3d_mrp_mlx README" (scope table: every sparse conv is (c, out, 3),
// stride 1, no padding -> submanifold; commit header: weight [O, kz, ky, kx, I],
// channels-last) and "pixal3d_mrp_mlx CLAUDE.md" ("Measured facts").
// Orientation reading: cross-correlation, as a dense Conv3d.
//
// Parallelism: OpenMP over output voxels for the neighbour lookups and the rows;
// the map is built single-threaded and only read afterwards.

#include <cstdint>
#include <unordered_map>
#include <vector>
#include <omp.h>

namespace {

constexpr int kOk = 0;
constexpr int kErrArg = -1;
constexpr int kErrCoordRange = -2;
constexpr int kErrDuplicate = -3;

inline uint64_t pack(int64_t b, int64_t z, int64_t y, int64_t x) {
  return (uint64_t(b) << 48) | (uint64_t(z) << 32) | (uint64_t(y) << 16) | uint64_t(x);
}

struct Map {
  std::unordered_map<uint64_t, int64_t> s;
  int status = kOk;
  int64_t bad_row = -1;
};

void build_map(const int32_t* coords, int64_t N, int32_t res, Map& m) {
  m.s.reserve(size_t(N) * 2 + 1);
  for (int64_t i = 0; i < N; ++i) {
    const int32_t b = coords[4 * i], z = coords[4 * i + 1], y = coords[4 * i + 2],
                  x = coords[4 * i + 3];
    if (b < 0 || b > 65534 || z < 0 || z >= res || y < 0 || y >= res || x < 0 || x >= res) {
      m.status = kErrCoordRange;
      m.bad_row = i;
      return;
    }
    auto ins = m.s.emplace(pack(b, z, y, x), i);
    if (!ins.second) {
      m.status = kErrDuplicate;
      m.bad_row = i;
      return;
    }
  }
}

inline int64_t lookup(const Map& m, int32_t res, int64_t b, int64_t z, int64_t y, int64_t x) {
  if (z < 0 || z >= res || y < 0 || y >= res || x < 0 || x >= res) return -1;
  auto it = m.s.find(pack(b, z, y, x));
  return it == m.s.end() ? -1 : it->second;
}

int set_threads(int nthreads) {
  if (nthreads > 0) omp_set_num_threads(nthreads);
  int used = 1;
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
  }
  return used;
}

}  // namespace

extern "C" {

// Number of OpenMP threads the next call will use (nthreads <= 0: the default).
int oracle_threads(int nthreads) { return set_threads(nthreads); }

// nbr int32 [N, 27] (-1 = absent). Returns 0, or -1 bad argument, -2 a coordinate
// out of range, -3 a duplicate coordinate; *bad_row receives the offending row.
int oracle_kernel_map(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                      int nthreads, int64_t* bad_row) {
  if (N < 0 || res < 1 || res > 65535 || (N > 0 && (!coords || !nbr))) return kErrArg;
  Map m;
  build_map(coords, N, res, m);
  if (bad_row) *bad_row = m.bad_row;
  if (m.status != kOk) return m.status;
  set_threads(nthreads);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; ++i) {
    const int64_t b = coords[4 * i], z = coords[4 * i + 1], y = coords[4 * i + 2],
                  x = coords[4 * i + 3];
    int k = 0;
    for (int dz = -1; dz <= 1; ++dz)
      for (int dy = -1; dy <= 1; ++dy)
        for (int dx = -1; dx <= 1; ++dx, ++k)
          nbr[27 * i + k] = int32_t(lookup(m, res, b, z + dz, y + dy, x + dx));
  }
  return kOk;
}

// out double [nrows, O] for the output rows listed in rows[] (each in [0, N)).
// feats float [N, I], weight float [O, 3, 3, 3, I], bias float [O] or NULL.
int oracle_forward_rows(const int32_t* coords, int64_t N, int32_t res, const float* feats,
                        int32_t I, const float* weight, int32_t O, const float* bias,
                        const int64_t* rows, int64_t nrows, double* out, int nthreads,
                        int64_t* bad_row) {
  if (N < 0 || res < 1 || res > 65535 || I < 1 || O < 1 || nrows < 0) return kErrArg;
  if (N > 0 && (!coords || !feats || !weight)) return kErrArg;
  if (nrows > 0 && (!rows || !out)) return kErrArg;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return kErrArg;
  Map m;
  build_map(coords, N, res, m);
  if (bad_row) *bad_row = m.bad_row;
  if (m.status != kOk) return m.status;
  set_threads(nthreads);
#pragma omp parallel
  {
    std::vector<double> acc(O);
#pragma omp for schedule(dynamic, 64)
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t i = rows[r];
      const int64_t b = coords[4 * i], z = coords[4 * i + 1], y = coords[4 * i + 2],
                    x = coords[4 * i + 3];
      for (int o = 0; o < O; ++o) acc[o] = bias ? double(bias[o]) : 0.0;
      for (int dz = -1; dz <= 1; ++dz)
        for (int dy = -1; dy <= 1; ++dy)
          for (int dx = -1; dx <= 1; ++dx) {
            const int64_t j = lookup(m, res, b, z + dz, y + dy, x + dx);
            if (j < 0) continue;
            const int tap = 9 * (dz + 1) + 3 * (dy + 1) + (dx + 1);
            const float* f = feats + j * int64_t(I);
            for (int o = 0; o < O; ++o) {
              const float* w = weight + (int64_t(o) * 27 + tap) * int64_t(I);
              double s = 0.0;
              for (int c = 0; c < I; ++c) s += double(w[c]) * double(f[c]);
              acc[o] += s;
            }
          }
      for (int o = 0; o < O; ++o) out[r * int64_t(O) + o] = acc[o];
    }
  }
  return kOk;
}

}  // extern "C"
