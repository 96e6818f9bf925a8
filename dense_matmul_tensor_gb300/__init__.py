"""GB300-native batched dense matrix product.

C[b] = alpha * op(A[b]) * op(B[b]) + beta * C[b] with bf16/fp16 inputs, fp32
accumulation on the tcgen05 tensor cores and fp32 or bf16 output, exposed
through the C ABI in ``include/bmm.h`` (``bmm_create`` / ``bmm_run`` /
``bmm_destroy``) and the thin binding in ``dense_matmul_tensor_gb300.bmm``.
"""
__all__ = ["bmm", "workloads", "build"]
