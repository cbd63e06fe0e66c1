"""CPU oracle of the W8A8 INT8 fused-MoE layer (test infrastructure only).

Only the tests, the smoke check and the bench's CPU-baseline leg import this
package; the product path never does, and this package imports nothing from
the product path."""
