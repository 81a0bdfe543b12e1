"""CPU oracle for the KV-cache block checksum.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the CPU-baseline legs of the benchmark, never by the product library.

* ``kvcs_oracle``: pure-Python exact-integer form (small inputs).
* ``c_oracle``: ctypes wrapper over the scalar C form in ``kvcs_oracle.c``
  (any size; also the timed CPU baseline).
"""
