"""fp64 CPU oracle for the attention forward -- test infrastructure, not the product path.

Only ``tests/``, the smoke check and the CPU-baseline leg of ``bench.py`` may import this
package.  The CUDA library neither imports it nor shares any code with it.
"""
