// tg_inst.cu - explicit instantiations of the GEMM kernel and its launcher.
// Compiled once per (TG_INST_F32, TG_INST_MODE) pair; MODE 0 dense, 1 grouped, 2 MoE.
#include "tg_launch.cuh"

#ifndef TG_INST_F32
#error "define TG_INST_F32 (0/1)"
#endif
#ifndef TG_INST_MODE
#error "define TG_INST_MODE (0/1/2)"
#endif

namespace tg {

template <class Cfg>
cudaError_t launch(const Params& p, int grid, cudaStream_t stream) {
    auto kern = &gemm_kernel<Cfg>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (Cfg::CTA_GROUP == 2) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (p.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <class Cfg>
cudaError_t resident_units(int* units) {
    auto kern = &gemm_kernel<Cfg>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (Cfg::CTA_GROUP == 1) {
        int per_sm = 0, dev = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NUM_THREADS, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        *units = per_sm * sms;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(units, kern, &cfg);
}

#define TG_INSTANTIATE(BN, CG, AMN, BMN, F32, MODE)                                                        \
    template cudaError_t launch<Config<BN, CG, AMN, BMN, F32, MODE>>(const Params&, int, cudaStream_t);   \
    template cudaError_t resident_units<Config<BN, CG, AMN, BMN, F32, MODE>>(int*);

#if TG_INST_MODE == 2
TG_FOR_EACH_MOE_TILE(TG_INSTANTIATE, (TG_INST_F32 != 0))
#else
TG_FOR_EACH_TILE(TG_INSTANTIATE, (TG_INST_F32 != 0), TG_INST_MODE)
#endif

}  // namespace tg
