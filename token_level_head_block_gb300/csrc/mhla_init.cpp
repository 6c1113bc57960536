// Host-side construction of the MHLA mixing matrix W from block-centre distances.
//
// Follows BlockDistanceConv of the MHLA module walkthrough (171host.com/767426.html,
// section 7): block centres at (index + 0.5) in block units, Euclidean distances
// between every pair, one of five distance -> weight transforms, then each column
// divided by its sum.  Extended from the listing's square 2-D grids to rectangular
// and 3-D grids by the same rule.  Arithmetic is double, rounded once to float;
// compile without floating-point contraction so every step rounds as written.
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/mhla.h"

namespace {

constexpr double kPi = 3.14159265358979323846;

int grid_blocks(const mhla_shape3_t* grid, const mhla_shape3_t* block, int64_t nb[3], int* ndim) {
  if (!grid || !block) return MHLA_ERR_INVALID_ARG;
  if (grid->ndim != block->ndim || (grid->ndim != 2 && grid->ndim != 3)) return MHLA_ERR_SHAPE;
  *ndim = grid->ndim;
  for (int a = 0; a < grid->ndim; ++a) {
    const int64_t g = grid->extent[a], b = block->extent[a];
    if (g <= 0 || b <= 0 || g % b != 0) return MHLA_ERR_SHAPE;
    nb[a] = g / b;
  }
  return MHLA_OK;
}

}  // namespace

extern "C" int64_t mhla_num_blocks(const mhla_shape3_t* grid, const mhla_shape3_t* block) {
  int64_t nb[3];
  int ndim = 0;
  const int rc = grid_blocks(grid, block, nb, &ndim);
  if (rc != MHLA_OK) return -static_cast<int64_t>(rc);
  int64_t M = 1;
  for (int a = 0; a < ndim; ++a) M *= nb[a];
  return M;
}

extern "C" mhla_status_t mhla_init_mixing(const mhla_shape3_t* grid, const mhla_shape3_t* block,
                                          int32_t transform, double local_thres, double exp_sigma,
                                          float* W_host, int64_t W_capacity) {
  if (!W_host) return MHLA_ERR_INVALID_ARG;
  if (transform < MHLA_TRANSFORM_LINEAR || transform > MHLA_TRANSFORM_LOCAL) return MHLA_ERR_INVALID_ARG;
  if (transform == MHLA_TRANSFORM_EXP && !(exp_sigma > 0.0)) return MHLA_ERR_INVALID_ARG;
  if (transform == MHLA_TRANSFORM_LOCAL && !(local_thres >= 0.0)) return MHLA_ERR_INVALID_ARG;
  int64_t nb[3];
  int ndim = 0;
  const int rc = grid_blocks(grid, block, nb, &ndim);
  if (rc != MHLA_OK) return static_cast<mhla_status_t>(rc);
  int64_t M = 1;
  for (int a = 0; a < ndim; ++a) M *= nb[a];
  if (M > (int64_t{1} << 15)) return MHLA_ERR_INVALID_ARG;  // M*M doubles must fit in memory
  if (W_capacity < M * M) return MHLA_ERR_INVALID_ARG;
  if (M == 1) {  // every transform column-normalises a single positive entry to 1
    W_host[0] = 1.0f;
    return MHLA_OK;
  }

  // Block centres, row-major block ids with the slowest axis first.
  std::vector<double> centre(static_cast<size_t>(M) * ndim);
  for (int64_t id = 0; id < M; ++id) {
    int64_t rem = id;
    for (int a = ndim - 1; a >= 0; --a) {
      centre[id * ndim + a] = static_cast<double>(rem % nb[a]) + 0.5;
      rem /= nb[a];
    }
  }
  std::vector<double> D(static_cast<size_t>(M) * M);
  double maxD = 0.0;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < M; ++j) {
      double s = 0.0;
      for (int a = 0; a < ndim; ++a) {
        const double diff = centre[i * ndim + a] - centre[j * ndim + a];
        s = s + diff * diff;
      }
      const double dist = std::sqrt(s);
      D[i * M + j] = dist;
      if (dist > maxD) maxD = dist;
    }

  std::vector<double> mat(static_cast<size_t>(M) * M);
  const double sigma_g = maxD / 3;
  for (size_t e = 0; e < mat.size(); ++e) {
    const double x = D[e];
    double y = 0.0;
    switch (transform) {
      case MHLA_TRANSFORM_LINEAR: y = 1.0 - x / maxD; break;
      case MHLA_TRANSFORM_COS: y = std::cos(x / maxD * kPi / 4); break;
      case MHLA_TRANSFORM_EXP: y = std::exp(-x / exp_sigma); break;
      case MHLA_TRANSFORM_GAUSSIAN: y = std::exp(-(x * x) / (2 * sigma_g * sigma_g)); break;
      default: y = (x <= local_thres) ? 1.0 : 0.0; break;
    }
    mat[e] = y;
  }
  // Column sums, accumulated from the top row down.
  std::vector<double> col(static_cast<size_t>(M), 0.0);
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < M; ++j) col[j] = col[j] + mat[i * M + j];
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < M; ++j) W_host[i * M + j] = static_cast<float>(mat[i * M + j] / col[j]);
  return MHLA_OK;
}
