"""Routed-expert MoE layer for GB300 (sm_103a): the C ABI of libmoe_route.so
and its thin Python binding. See include/moe_route.h for the contract."""
from ._lib import (EXPORTED, LIB_PATH, MOE_BF16, MOE_POLICY_FETCH_ALL, MOE_POLICY_FIRST_CHOICE,
                   MOE_POLICY_THRESHOLD, MOE_ERR_BAD_INDEX, MOE_ERR_CUDA,
                   MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED,
                   MOE_ERR_WORKSPACE, MOE_F16, MOE_F32, MOE_OK, MOE_OP_DECODE, MOE_OP_LAYER,
                   MOE_OP_LAYER_RESIDENT, MOE_OP_PREFILL, MOE_OP_PREROUTE, MOE_OP_ROUTE,
                   MOE_OP_SHARED, ExpertCache, Experts, MoeError, Prerouter, Router, Shared,
                   moe_cache_plan, moe_cache_workspace_bytes, moe_cached_layer, moe_pool_fetch,
                   StageTable, moe_stage_plan, moe_stage_prediction,
                   moe_check_status, moe_decode, moe_layer, moe_layer_noalloc, moe_layer_resident,
                   moe_layer_stack, moe_layer_stack_resident, moe_prefill, moe_preroute, moe_replay, moe_route,
                   moe_set_wait_limit, moe_shared_lora, moe_substitute,
                   moe_workspace_bytes, status_string, workspace)

__all__ = [n for n in dir() if not n.startswith("_")]
