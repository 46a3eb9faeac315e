// The standalone Forecast projection launch: one CTA per tile of 8 rows x kProjSeqs sequences (the
// computation is project_rows in project_body.cuh).
#include "project_body.cuh"

namespace sparda {

__global__ void __launch_bounds__(kProjThreads) forecast_project_kernel(const ProjectArgs a) {
  __shared__ ProjShared sh;
  grid_dep_launch();                   // the selector may start streaming compressed keys
  project_rows(a, blockIdx.x, blockIdx.y, sh, 1);
}

void launch_forecast_project(const ProjectArgs& a, cudaStream_t s) {
  dim3 grid(a.rows / 8, (a.batch + kProjSeqs - 1) / kProjSeqs);
  forecast_project_kernel<<<grid, kProjThreads, 0, s>>>(a);
}

}  // namespace sparda
