// tc.cu -- tcgen05/TMEM tensor-core single-pass path (sm_103a).
#include "common.cuh"

namespace la {

bool tc_supported(const Problem &p, int num_sms)
{
    (void)p;
    (void)num_sms;
    return false;
}

int tc_plan(const Problem &p, int num_sms, la_plan_info *info)
{
    (void)p;
    (void)num_sms;
    (void)info;
    return LA_ERR_UNSUPPORTED;
}

int tc_launch(const Problem &p, int num_sms)
{
    (void)p;
    (void)num_sms;
    return LA_ERR_UNSUPPORTED;
}

}  // namespace la
