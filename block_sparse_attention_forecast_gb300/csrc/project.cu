// The standalone Forecast projection launch; the computation is in project_body.cuh.
#include "project_body.cuh"

namespace sparda {

__global__ void __cluster_dims__(1, kProjSplit, 1) __launch_bounds__(kProjThreads)
    forecast_project_kernel(const ProjectArgs a) {
  __shared__ ProjShared sh;
  grid_dep_launch();                   // the selector may start streaming compressed keys
  project_cta(a, blockIdx.x, blockIdx.y, blockIdx.z, sh);
}

void launch_forecast_project(const ProjectArgs& a, cudaStream_t s) {
  dim3 grid(a.rows / 8, kProjSplit, (a.batch + 15) / 16);
  forecast_project_kernel<<<grid, kProjThreads, 0, s>>>(a);
}

}  // namespace sparda
