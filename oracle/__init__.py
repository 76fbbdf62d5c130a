"""CPU oracle for the mixture-of-experts layer step.

Test infrastructure only: the tests, the package smoke check and the CPU
baseline leg of the benchmark are its only users.  The CUDA library never
imports it.
"""
